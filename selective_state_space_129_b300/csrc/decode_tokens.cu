// K consecutive decode tokens of the Mamba-3 scan in one launch, the state
// kept on chip between them.
//
// For every (batch, head) and t = 0 .. K-1 the step is the decode recurrence
// (Prop. 1 and the rotation, sec. 4.1 and 4.2 of
// "MAMBA-3: IMPROVED SEQUENCE MODELING USING STATE SPACE PRINCIPLES" (aipaper.cc); MIMO
// rank R, sec. 3 of "Mamba-3: Improved Sequence Modeling using State Space Principles" (papernotes.org)):
//   h_t = alpha_t Rot(Delta_t theta_t) (h_{t-1} + beta_hat_t B_{t-1} x_{t-1}^T)
//         + gamma_t B_t x_t^T,        y_t = C_t^T h_t
// where B_{t-1}, x_{t-1} is the previous token of the block (the caller's
// B_prev / x_prev for t = 0). Written once per token, the step reads and
// writes the N x P fp32 state every token; here the state is read once, held
// in registers for the K tokens and written once, so that its HBM traffic per
// token falls by K (the multi-token decode of speculative or batched-token
// serving).
//
// One CTA per (batch, head), 256 threads. A work item is one rotating row pair
// (2k, 2k+1) times four consecutive columns; thread tid owns items
// tid + 256 m (m < 4), so the whole state (N P <= 8192) sits in 32 registers
// per thread. The token activations of the block (x, B, C, theta, dt, lambda,
// the biases, B_prev, x_prev) are copied into shared memory once, with 16-byte
// asynchronous copies issued while the state loads are in flight. The
// coefficient rows do not depend on the state, so the CTA forms those of a
// window of W tokens (as many as shared memory holds, often all K) in one
// parallel pass, with the rotation folded into the B_prev term,
// alpha Rot(beta_hat (B_prev + bias) x_prev^T) = (alpha Rot beta_hat (B_prev +
// bias)) x_prev^T, so that each item computes
//   h' = alpha Rot h + U (x_prev | x)^T,
//   U  = [alpha Rot beta_hat (B_prev + bias) | gamma (B + bias)]   (N x 2R).
// The tokens of a window then run back to back with no barrier between them:
// a step is bound by its instruction count (the state no longer streams), so
// every product is a packed two-lane FMA over a pair of columns, its
// coefficient operand a (v, v) pair stored twice in the tables, and the
// partial y are folded by warp shuffles into a per-token table that is summed
// at the end of the window.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace m3 {
namespace {

constexpr int kTThreads = 256;
constexpr int kTWarps = kTThreads / 32;
constexpr int kTItems = 4;  // items per thread: a state of at most 1024 items (N P <= 8192)

// CTAs per SM the kernel is built for: three at R <= 2 (at most 85 registers
// a thread; the R = 4 step needs more), two at R = 4. The token window is
// sized so that their shared memory fits too.
__host__ __device__ constexpr int tok_ctas_per_sm(int R) { return R <= 2 ? 3 : 2; }
__host__ __device__ constexpr uint64_t tok_smem_keep(int R) {
  return R <= 2 ? 72 * 1024 : 110 * 1024;
}
constexpr uint64_t kTokSmemMax = 200 * 1024;

__host__ __device__ inline uint32_t tup16(uint64_t v) { return (uint32_t)((v + 15) & ~uint64_t(15)); }

// Byte offsets of the block's activations in shared memory (K tokens), then
// the coefficient tables and the partial-y table (floats).
struct TokLayout {
  uint32_t x, B, C, th, bb, cb, xp, Bp, dt, lm;  // bases; per-token strides below
  uint32_t sx, sbc, sth;                         // per-token strides of x, B / C, theta
  uint32_t coef, scoef;                          // coefficient tables, per-token stride
  uint32_t yred, syred;                          // partial-y tables, per-token stride
  uint32_t win, bytes;                           // tokens per window, total bytes
};

inline TokLayout tok_layout(const TokensArgs& a, int act) {
  const uint64_t N = a.N, P = a.P, R = a.R, K = a.K;
  TokLayout L{};
  L.sx = tup16(P * R * act);
  L.sbc = tup16(N * R * act);
  L.sth = tup16(N / 2 * 4);
  uint64_t o = 0;
  L.x = (uint32_t)o; o += K * L.sx;
  L.B = (uint32_t)o; o += K * L.sbc;
  L.C = (uint32_t)o; o += K * L.sbc;
  L.th = (uint32_t)o; o += K * L.sth;
  L.bb = (uint32_t)o; o += a.B_bias ? tup16(N * R * 4) : 0;
  L.cb = (uint32_t)o; o += a.C_bias ? tup16(N * R * 4) : 0;
  L.xp = (uint32_t)o; o += a.x_prev ? L.sx : 0;
  L.Bp = (uint32_t)o; o += a.B_prev ? L.sbc : 0;
  L.dt = (uint32_t)o; o += tup16(K * 4);
  L.lm = (uint32_t)o; o += tup16(K * 4);
  // per token: U pairs [N][2R][2], C + bias pairs [N][R][2], and per row pair
  // (ac, ac, as, as, -as, -as, 0, 0) with ac, as = alpha (cos, sin)
  L.scoef = (uint32_t)((6 * N * R + 4 * N) * 4);
  L.syred = (uint32_t)((uint64_t)kTWarps * R * (P + 4) * 4);
  const uint64_t per = (uint64_t)L.scoef + L.syred;
  const uint64_t keep = tok_smem_keep((int)R);
  uint64_t w = o < keep ? (keep - o) / per : 0;
  if (w < 1) w = 1;
  if (w > K) w = K;
  L.win = (uint32_t)w;
  L.coef = (uint32_t)o; o += w * L.scoef;
  L.yred = (uint32_t)o; o += w * L.syred;
  L.bytes = (uint32_t)(o < 0xffffffffull ? o : 0xffffffffull);
  return L;
}

// Every thread copies its share of a block of `bytes` (a multiple of 16) with
// 16-byte asynchronous copies; completion is awaited with cp_async_wait_all.
__device__ __forceinline__ void copy_block(uint8_t* dst, const void* src, uint32_t bytes, int tid) {
  const uint8_t* s = static_cast<const uint8_t*>(src);
  for (uint32_t i = 16u * tid; i < bytes; i += 16u * kTThreads) ptx::cp_async16(dst + i, s + i);
}

// The 4 x R activations of one column quad from shared memory.
template <typename T, int R>
__device__ __forceinline__ void ld_quad_t(const T* p, float (&v)[4][R]) {
#pragma unroll
  for (int i = 0; i < 4 * R; ++i) v[i / R][i % R] = ld_act(p + i);
}

template <typename T, int R>
__global__ void __launch_bounds__(kTThreads, tok_ctas_per_sm(R))
    decode_tokens_kernel(TokensArgs a, TokLayout L) {
  extern __shared__ __align__(16) uint8_t sm[];
  const int K = (int)a.K, N = (int)a.N, P = (int)a.P, K2 = N / 2, PQ = P / 4, H = (int)a.H;
  const int hpg = (int)(a.H / a.G);
  const int64_t u = blockIdx.x, b = u / H, h = u % H, g = h / hpg;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = tid % PQ;  // this thread's column quad (PQ divides 32)
  const int items = K2 * PQ;
  const bool has_prev = a.B_prev != nullptr;
  const int64_t NR = (int64_t)N * R, PR = (int64_t)P * R;

  // 1. this thread's state items into registers (in flight during the copies)
  float* gst = a.state + u * N * P;
  float4 h0[kTItems], h1[kTItems];
#pragma unroll
  for (int m = 0; m < kTItems; ++m) {
    const int it = tid + kTThreads * m;
    if (it < items) {
      const int kq = it / PQ;
      h0[m] = *reinterpret_cast<const float4*>(gst + (2 * kq) * P + 4 * q);
      h1[m] = *reinterpret_cast<const float4*>(gst + (2 * kq + 1) * P + 4 * q);
    } else {
      h0[m] = h1[m] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }

  // 2. the block's activations into shared memory
  const T* gx = static_cast<const T*>(a.x);
  const T* gB = static_cast<const T*>(a.B);
  const T* gC = static_cast<const T*>(a.C);
  for (int t = 0; t < K; ++t) {
    const int64_t bt = b * K + t;
    copy_block(sm + L.x + t * L.sx, gx + (bt * H + h) * PR, (uint32_t)(PR * sizeof(T)), tid);
    copy_block(sm + L.B + t * L.sbc, gB + (bt * a.G + g) * NR, (uint32_t)(NR * sizeof(T)), tid);
    copy_block(sm + L.C + t * L.sbc, gC + (bt * a.G + g) * NR, (uint32_t)(NR * sizeof(T)), tid);
    copy_block(sm + L.th + t * L.sth, a.theta + (bt * a.G + g) * K2, (uint32_t)K2 * 4, tid);
  }
  if (a.B_bias) copy_block(sm + L.bb, a.B_bias + h * NR, (uint32_t)NR * 4, tid);
  if (a.C_bias) copy_block(sm + L.cb, a.C_bias + h * NR, (uint32_t)NR * 4, tid);
  if (has_prev) {
    copy_block(sm + L.xp, static_cast<const T*>(a.x_prev) + u * PR, (uint32_t)(PR * sizeof(T)), tid);
    copy_block(sm + L.Bp, static_cast<const T*>(a.B_prev) + (b * a.G + g) * NR,
               (uint32_t)(NR * sizeof(T)), tid);
  }
  float* sdt = reinterpret_cast<float*>(sm + L.dt);
  float* slm = reinterpret_cast<float*>(sm + L.lm);
  for (int t = tid; t < K; t += kTThreads) {
    sdt[t] = a.dt[(b * K + t) * H + h];
    slm[t] = a.lam[(b * K + t) * H + h];
  }
  const float A_h = a.A[h];
  ptx::cp_async_wait_all();
  __syncthreads();

  const float* sbb = reinterpret_cast<const float*>(sm + L.bb);
  const float* scb = reinterpret_cast<const float*>(sm + L.cb);

  // y of token t from its partial-y table yred[(w 4R + c R + r)(PQ + 1) + q]
  auto final_sum = [&](int t, const float* yred) {
    T* out = static_cast<T*>(a.out) + (((int64_t)b * K + t) * H + h) * PR;
    for (int i = tid; i < PR; i += kTThreads) {
      const int pp = i / R, r = i - pp * R;
      const int at = ((pp & 3) * R + r) * (PQ + 1) + (pp >> 2);
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < kTWarps; ++w) acc += yred[w * 4 * R * (PQ + 1) + at];
      st_act(out + i, acc);
    }
  };

  // row pair of each of this thread's items (-1: none), fixed for the call
  int kqs[kTItems];
#pragma unroll
  for (int m = 0; m < kTItems; ++m) {
    const int it = tid + kTThreads * m;
    kqs[m] = it < items ? it / PQ : -1;
  }
  const int ybase = warp * 4 * R * (PQ + 1) + q;  // this lane's slot in a partial-y table

  for (int t0 = 0; t0 < K; t0 += (int)L.win) {
    const int nw = min((int)L.win, K - t0);
    // 3. coefficient tables of tokens t0 .. t0 + nw - 1 (token t's B_prev is
    // token t-1 of the block): entry e = (token, row pair kq, rank r)
    for (int e = tid; e < nw * K2 * R; e += kTThreads) {
      const int tw = e / (K2 * R), e2 = e - tw * K2 * R, kq = e2 / R, r = e2 - kq * R;
      const int t = t0 + tw;
      const float d = sdt[t], lm = slm[t];
      const float alpha = expf(d * A_h);
      const float gamma = lm * d, bhat = (1.f - lm) * d;
      const T* sB = reinterpret_cast<const T*>(sm + L.B + t * L.sbc);
      const T* sC = reinterpret_cast<const T*>(sm + L.C + t * L.sbc);
      const T* sBp = reinterpret_cast<const T*>(t > 0 ? sm + L.B + (t - 1) * L.sbc : sm + L.Bp);
      const float* sth = reinterpret_cast<const float*>(sm + L.th + t * L.sth);
      float2* ud = reinterpret_cast<float2*>(sm + L.coef + tw * L.scoef);  // [N][2R] pairs
      float2* cd = ud + 2 * NR;                                           // [N][R] pairs
      float4* rd = reinterpret_cast<float4*>(cd + NR);                    // [K2][2]
      float sn, cs;
      __sincosf(wrap_angle(d * sth[kq]), &sn, &cs);
      const float ac = alpha * cs, as = alpha * sn;
      const int i0 = 2 * kq * R + r, i1 = i0 + R;  // (row 2kq, r), (row 2kq + 1, r)
      const float bb0 = a.B_bias ? sbb[i0] : 0.f, bb1 = a.B_bias ? sbb[i1] : 0.f;
      const float cb0 = a.C_bias ? scb[i0] : 0.f, cb1 = a.C_bias ? scb[i1] : 0.f;
      float u0 = 0.f, u1 = 0.f;
      if (t > 0 || has_prev) {
        const float p0 = bhat * (ld_act(sBp + i0) + bb0), p1 = bhat * (ld_act(sBp + i1) + bb1);
        u0 = fmaf(ac, p0, -as * p1);
        u1 = fmaf(as, p0, ac * p1);
      }
      const float g0 = gamma * (ld_act(sB + i0) + bb0), g1 = gamma * (ld_act(sB + i1) + bb1);
      float2* U0 = ud + 2 * kq * 2 * R;  // row 2kq: [rotated B_prev term | B term], then row 2kq + 1
      U0[r] = make_float2(u0, u0);
      U0[R + r] = make_float2(g0, g0);
      U0[2 * R + r] = make_float2(u1, u1);
      U0[3 * R + r] = make_float2(g1, g1);
      const float c0 = ld_act(sC + i0) + cb0, c1 = ld_act(sC + i1) + cb1;
      cd[i0] = make_float2(c0, c0);
      cd[i1] = make_float2(c1, c1);
      if (r == 0) {
        rd[2 * kq] = make_float4(ac, ac, as, as);
        rd[2 * kq + 1] = make_float4(-as, -as, 0.f, 0.f);
      }
    }
    __syncthreads();

    // 4. the window's tokens, back to back
    for (int tw = 0; tw < nw; ++tw) {
      const int t = t0 + tw;
      const float4* U4 = reinterpret_cast<const float4*>(sm + L.coef + tw * L.scoef);  // R per row
      const float4* C4 = U4 + 2 * NR / 2;   // rows 2kq, 2kq + 1: R float4
      const float4* R4 = C4 + NR / 2;       // 2 per row pair
      float* yred = reinterpret_cast<float*>(sm + L.yred + tw * L.syred);
      const bool prev = t > 0 || has_prev;
      // X[cp][j]: (x_prev | x)[ranks j] of the column pair (4q + 2cp, 4q + 2cp + 1)
      float2 X[2][2 * R];
      {
        float xr[4][R], xpr[4][R];
        ld_quad_t<T, R>(reinterpret_cast<const T*>(sm + L.x + t * L.sx) + 4 * q * R, xr);
        if (prev) {
          const T* sxp = reinterpret_cast<const T*>(t > 0 ? sm + L.x + (t - 1) * L.sx : sm + L.xp);
          ld_quad_t<T, R>(sxp + 4 * q * R, xpr);
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int r = 0; r < R; ++r) xpr[c][r] = 0.f;
        }
#pragma unroll
        for (int cp = 0; cp < 2; ++cp)
#pragma unroll
          for (int r = 0; r < R; ++r) {
            X[cp][r] = make_float2(xpr[2 * cp][r], xpr[2 * cp + 1][r]);
            X[cp][R + r] = make_float2(xr[2 * cp][r], xr[2 * cp + 1][r]);
          }
      }
      float2 Y[2][R];
#pragma unroll
      for (int cp = 0; cp < 2; ++cp)
#pragma unroll
        for (int r = 0; r < R; ++r) Y[cp][r] = make_float2(0.f, 0.f);
#pragma unroll
      for (int m = 0; m < kTItems; ++m) {
        const int kq = kqs[m];
        if (kq >= 0) {
          const float4 ra = R4[2 * kq], rb = R4[2 * kq + 1];
          const float2 ac2 = make_float2(ra.x, ra.y), as2 = make_float2(ra.z, ra.w);
          const float2 nas2 = make_float2(rb.x, rb.y);
          float4 cw[R];  // C pairs of rows 2kq (first R / 2) and 2kq + 1
#pragma unroll
          for (int j = 0; j < R; ++j) cw[j] = C4[kq * R + j];
          const float2* cpair = reinterpret_cast<const float2*>(cw);  // [2][R]
          float2 n0[2], n1[2];
#pragma unroll
          for (int cp = 0; cp < 2; ++cp) {
            const float2 a0 = cp ? make_float2(h0[m].z, h0[m].w) : make_float2(h0[m].x, h0[m].y);
            const float2 a1 = cp ? make_float2(h1[m].z, h1[m].w) : make_float2(h1[m].x, h1[m].y);
            n0[cp] = ptx::fma2(ac2, a0, ptx::mul2(nas2, a1));
            n1[cp] = ptx::fma2(ac2, a1, ptx::mul2(as2, a0));
          }
#pragma unroll
          for (int j = 0; j < R; ++j) {  // U pairs 2j, 2j + 1 of rows 2kq and 2kq + 1
            const float4 w0 = U4[(2 * kq) * R + j], w1 = U4[(2 * kq + 1) * R + j];
#pragma unroll
            for (int cp = 0; cp < 2; ++cp) {
              n0[cp] = ptx::fma2(make_float2(w0.x, w0.y), X[cp][2 * j], n0[cp]);
              n0[cp] = ptx::fma2(make_float2(w0.z, w0.w), X[cp][2 * j + 1], n0[cp]);
              n1[cp] = ptx::fma2(make_float2(w1.x, w1.y), X[cp][2 * j], n1[cp]);
              n1[cp] = ptx::fma2(make_float2(w1.z, w1.w), X[cp][2 * j + 1], n1[cp]);
            }
          }
          h0[m] = make_float4(n0[0].x, n0[0].y, n0[1].x, n0[1].y);
          h1[m] = make_float4(n1[0].x, n1[0].y, n1[1].x, n1[1].y);
#pragma unroll
          for (int cp = 0; cp < 2; ++cp)
#pragma unroll
            for (int r = 0; r < R; ++r)
              Y[cp][r] = ptx::fma2(cpair[r], n0[cp], ptx::fma2(cpair[R + r], n1[cp], Y[cp][r]));
        }
      }
      // lanes with the same column quad fold by shuffles; the warps' partials
      // go to this token's table
      float yp[4][R];
#pragma unroll
      for (int cp = 0; cp < 2; ++cp)
#pragma unroll
        for (int r = 0; r < R; ++r) {
          yp[2 * cp][r] = Y[cp][r].x;
          yp[2 * cp + 1][r] = Y[cp][r].y;
        }
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int r = 0; r < R; ++r)
          for (int o = PQ; o < 32; o <<= 1) yp[c][r] += __shfl_xor_sync(0xffffffffu, yp[c][r], o);
      if (lane < PQ) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int r = 0; r < R; ++r) yred[ybase + (c * R + r) * (PQ + 1)] = yp[c][r];
      }
    }
    // the window's outputs; the next window's tables and partials are
    // written after the next barrier, which every thread reaches after these
    __syncthreads();
    for (int tw = 0; tw < nw; ++tw)
      final_sum(t0 + tw, reinterpret_cast<const float*>(sm + L.yred + tw * L.syred));
  }

  // 5. the state back, once
#pragma unroll
  for (int m = 0; m < kTItems; ++m) {
    const int kq = kqs[m];
    if (kq >= 0) {
      *reinterpret_cast<float4*>(gst + (2 * kq) * P + 4 * q) = h0[m];
      *reinterpret_cast<float4*>(gst + (2 * kq + 1) * P + 4 * q) = h1[m];
    }
  }
}

template <typename T>
cudaError_t launch_t(const TokensArgs& a, cudaStream_t s) {
  const TokLayout L = tok_layout(a, (int)sizeof(T));
  const dim3 grid((unsigned)(a.batch * a.H));
  cudaError_t e = cudaSuccess;
  switch (a.R) {
    case 1:
      e = cudaFuncSetAttribute(decode_tokens_kernel<T, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.bytes);
      if (e == cudaSuccess) decode_tokens_kernel<T, 1><<<grid, kTThreads, L.bytes, s>>>(a, L);
      break;
    case 2:
      e = cudaFuncSetAttribute(decode_tokens_kernel<T, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.bytes);
      if (e == cudaSuccess) decode_tokens_kernel<T, 2><<<grid, kTThreads, L.bytes, s>>>(a, L);
      break;
    case 4:
      e = cudaFuncSetAttribute(decode_tokens_kernel<T, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.bytes);
      if (e == cudaSuccess) decode_tokens_kernel<T, 4><<<grid, kTThreads, L.bytes, s>>>(a, L);
      break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

// Shapes the kernel takes: whole column quads with P/4 dividing a warp, the
// state in at most kTItems items per thread, 16-byte vectors for every
// per-token block, and the block's activations in one CTA's shared memory.
bool tokens_supported(const TokensArgs& a, int act) {
  const int64_t N = a.N, P = a.P, R = a.R;
  if (!(R == 1 || R == 2 || R == 4)) return false;
  if (P < 4 || P % 4 != 0 || 32 % (P / 4) != 0) return false;
  if (N < 2 || N % 2 != 0 || (N / 2) * (P / 4) > (int64_t)kTThreads * kTItems) return false;
  if ((P * R * act) % 16 || (N * R * act) % 16 || (N / 2 * 4) % 16) return false;
  if ((a.B_bias || a.C_bias) && (N * R * 4) % 16) return false;
  if (a.K < 1 || a.K > 4096) return false;
  return tok_layout(a, act).bytes <= kTokSmemMax;
}

cudaError_t launch_decode_tokens(const TokensArgs& a, bool bf16, cudaStream_t s) {
  if (tokens_mma_ok(a, bf16)) return launch_tokens_mma(a, s);
  return bf16 ? launch_t<__nv_bfloat16>(a, s) : launch_t<float>(a, s);
}

}  // namespace m3
