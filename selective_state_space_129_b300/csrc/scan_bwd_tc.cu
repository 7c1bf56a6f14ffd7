// Backward pass of the Mamba-3 scan on the tensor cores: the gradients of
// <y, dy> + <h_final, d_final> for a prefill from a zero state, bf16
// activations, P = 64, N in {64, 128}, R in {1, 2, 4}.
//
// Forward (Prop. 1 and the rotation, sec. 4.1 and 4.2 of "MAMBA-3: IMPROVED
// SEQUENCE MODELING USING STATE SPACE PRINCIPLES" (aipaper.cc); MIMO rank R,
// sec. 3 of "Mamba-3: Improved Sequence Modeling using State Space
// Principles" (papernotes.org)), written per chunk of Q = 64 / R tokens in the
// chunk's own rotation frame. With chunk-local sums Lam_t = sum_{u<=t} dt_u A
// and Phi_t[k] = sum_{u<=t} dt_u theta_u[k] (from the chunk's first token),
// Bt_t = Rot(-Phi_t)(B_t + bias), Ct_t likewise, and H_in the explicit-frame
// state entering the chunk (with the pending trapezoid term of its first token):
//   y_t   = e^{Lam_t} Ct_t^T H_in + sum_{s<=t} W_ts (Ct_t . Bt_s) x_s,
//   W_ts  = e^{Lam_t - Lam_s} (gamma_s + [s<t] bhat_{s+1}),
//   H_out = Rot(Phi_end) (e^{Lam_end} H_in + sum_s w_s Bt_s x_s^T),
//   w_s   = e^{Lam_end - Lam_s} (gamma_s + bhat_{s+1})
// (bhat of the token after the chunk; 0 past the end). Flattening (token, rank)
// into QR = 64 rows, S = Ct Bt^T, P = S o W and Y = P X + diag(e^Lam) Ct H_in
// is the chunked form of the scan (the papernotes.org page named above,
// sec. 1; SSD form Y = (L o C B^T) X).
//
// Backward, per chunk, with dG = Rot(-Phi_end) dH_out (dH_out = d_final for
// the last chunk) and H_in from a forward pass over the chunk boundaries:
//   dP = dY X^T,  dS = dP o W,  dW_ts = sum over the rank block of S o dP
//   dX  = P^T dY + diag(w) Bt dG
//   dCt = dS Bt + diag(e^Lam) dY H_in^T,     dBt = dS^T Ct + diag(w) X dG^T
//   dH_in = e^{Lam_end} dG + Ct^T diag(e^Lam) dY
//   d e^{Lam_t} = rows of Ct . (dY H_in^T),  dw_s = rows of Bt . (X dG^T)
// then the decay, trapezoid and rotation gradients:
//   dl_u = sum_{s<u<=t} dW_ts W_ts + sum_{t>=u} d(e^Lam_t) e^Lam_t
//          + sum_{s<u} dw_s w_s + e^{Lam_end} <dG, H_in>      (l_u = dt_u A)
//   (the first sum is the exclusive prefix over v < u of column minus row
//   sums of dW o W), dgamma_s, dbhat_{s+1} from column sums of dW o e^{Lam_t -
//   Lam_s} and from dw_s; dB = Rot(Phi_t) dBt, dPhi_t = sum_r (dBt_0 Bt_1 -
//   dBt_1 Bt_0) + the same for C + (at the chunk's last token) the rotation at
//   its end; dphi_u = sum_{t>=u} dPhi_t within the chunk.
//
// Three launches:
//   bwd_parts  one CTA per chunk: the chunk's contributions sum_s w_s Bt_s x_s^T
//              and Ct^T diag(e^Lam) dY to the two state recurrences, and the
//              chunk's Lam_end and Phi_end;
//   bwd_scan   per (b, h, pair, column): the forward recurrence over chunks
//              (H_in of every chunk) and the reverse one (dG of every chunk),
//              elementwise, with the chunk-end rotation and decay gradients;
//   bwd_chunk  one CTA per chunk: everything else.
// Every contraction is mma.sync m16n8k8 TF32 (fp32 accumulation) from fp32
// tiles in shared memory (x and dy are bf16 and exact in TF32). Gradients shared
// by heads, batch rows or tokens (dB, dC, dtheta, dA, the biases, and ddt /
// dlambda, which the next chunk's boundary term also adds to) are accumulated
// with atomics, so their last bits vary between runs.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace m3 {
namespace {

constexpr int kBT = 512;  // threads of the chunk kernels
constexpr int kRows = 64;  // flattened (token, rank) rows per chunk
constexpr int kPd = 64;    // head dim
constexpr int kSX = kPd + 4;  // word stride of the [64][P] tiles and of the [N][P] state tile

template <int R, int NS>
struct BCfg {
  static constexpr int Q = kRows / R;
  static constexpr int K2 = NS / 2;
  static constexpr int SB = NS + 4;   // word stride of the [64][N] tiles
  // row pitch (in (cos, sin) pairs) of the rotation table: 8 words mod 32, so
  // that the rotation backward's reads of 4 tokens x 4 pairs per half-warp
  // fall on 32 different banks
  static constexpr int RP = K2 + 4;
  static constexpr int TG = kBT / K2;  // token groups of the fold
  static constexpr int TPG = Q / TG;   // tokens per fold thread
  static_assert(TPG >= 1 && Q % TG == 0, "token groups must divide the chunk");
};

// Per-token values of one chunk (index t < Q; bh has one more entry, the
// token after the chunk).
struct TokTab {
  float lc[kRows];   // Lam_t, chunk-local inclusive sum of dt A
  float dt[kRows], lm[kRows], gam[kRows];
  float bh[kRows + 1];
  float w[kRows], el[kRows];
  float dtn, lmn;    // dt and lambda of the token after the chunk (0 past the end)
};

__device__ __forceinline__ float tf32r(float v) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
  return __uint_as_float(r);
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// acc[nt] += A x B with both operands stored k-major: A[m][k] at A[k SA + m]
// (rows m0 .. m0+15) and B[k][n] at B[k SBS + n] (columns n0 + 8 nt ..), fp32
// (TF32-rounded) in shared memory; each fragment word is loaded alone.
template <int NT, int K, int SA, int SBS>
__device__ __forceinline__ void wgemm_kk(float (&acc)[NT][4], const float* A, int m0,
                                         const float* B, int n0, int lane) {
  const int g = lane >> 2, tq = lane & 3;
  const float* ap = A + tq * SA + m0 + g;
  const float* bp = B + tq * SBS + n0 + g;
#pragma unroll
  for (int k0 = 0; k0 < K; k0 += 8) {
    const uint32_t a0 = __float_as_uint(ap[k0 * SA]);
    const uint32_t a1 = __float_as_uint(ap[k0 * SA + 8]);
    const uint32_t a2 = __float_as_uint(ap[(k0 + 4) * SA]);
    const uint32_t a3 = __float_as_uint(ap[(k0 + 4) * SA + 8]);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const uint32_t b0 = __float_as_uint(bp[k0 * SBS + 8 * nt]);
      const uint32_t b1 = __float_as_uint(bp[(k0 + 4) * SBS + 8 * nt]);
      mma_tf32(acc[nt], a0, a1, a2, a3, b0, b1);
    }
  }
}

__device__ __forceinline__ void ldm4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                     uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Row order of the per-chunk kernel's tiles that serve as B operands: within
// each block of 8 rows, row k is stored at 2 (k % 4) + k / 4 (so rows 0..7 at
// 0, 2, 4, 6, 1, 3, 5, 7). A B fragment's two k rows, tq and tq + 4, then sit
// side by side at 2 tq, 2 tq + 1, and its word loads from a [k][n] tile (word
// stride 4 mod 32) fall on 32 different banks; ldmatrix takes any row order.
__device__ __forceinline__ int prow(int k) { return (k & ~7) | ((k & 3) << 1) | ((k >> 2) & 1); }

// acc[nt] += A (rows m0 .. m0+15 of a row-major [m][k] fp32 tile, word stride
// SA, at shared address a_tile) x B (K x 8 NT, columns n0 + 8 nt ..). The A
// fragments come by ldmatrix: an 8 x 4 block of 32-bit words is the b16 8 x 8
// matrix whose distribution (thread t: row t / 4, word t % 4) is the TF32
// fragment's. BL: B is stored [n][k] (word stride SBS, at b_tile) and comes by
// ldmatrix, two n-tiles at a time; else B is stored [k][n] (Bp) and each
// fragment word is loaded alone. B's rows are in prow order; A's rows too
// when PA.
template <int NT, int K, int SA, int SBS, bool BL, bool PA>
__device__ __forceinline__ void wgemm_l(float (&acc)[NT][4], uint32_t a_tile, int m0,
                                        uint32_t b_tile, const float* Bp, int n0, int lane) {
  const int g = lane >> 2, tq = lane & 3, mi = lane >> 3, rr = lane & 7;
  const int ra = m0 + rr + 8 * (mi & 1);
  const uint32_t a_lane = a_tile + 4u * (uint32_t)((PA ? prow(ra) : ra) * SA + 4 * (mi >> 1));
  const uint32_t b_lane = b_tile + 4u * (uint32_t)(prow(n0 + rr + 8 * (mi >> 1)) * SBS + 4 * (mi & 1));
  // k rows k0 + tq and k0 + tq + 4 are stored at k0 + 2 tq and k0 + 2 tq + 1
  const float* bp = Bp + 2 * tq * SBS + n0 + g;
#pragma unroll
  for (int k0 = 0; k0 < K; k0 += 8) {
    uint32_t a0, a1, a2, a3;
    ldm4(a_lane + 4u * k0, a0, a1, a2, a3);
    if constexpr (BL) {
      static_assert(NT % 2 == 0, "n-tiles come in pairs");
#pragma unroll
      for (int nt = 0; nt < NT; nt += 2) {
        uint32_t b0, b1, b2, b3;
        ldm4(b_lane + 4u * (8 * nt * SBS + k0), b0, b1, b2, b3);
        mma_tf32(acc[nt], a0, a1, a2, a3, b0, b1);
        mma_tf32(acc[nt + 1], a0, a1, a2, a3, b2, b3);
      }
    } else {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint32_t b0 = __float_as_uint(bp[k0 * SBS + 8 * nt]);
        const uint32_t b1 = __float_as_uint(bp[(k0 + 1) * SBS + 8 * nt]);
        mma_tf32(acc[nt], a0, a1, a2, a3, b0, b1);
      }
    }
  }
}

template <int NT>
__device__ __forceinline__ void zero_acc(float (&acc)[NT][4]) {
#pragma unroll
  for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
}

// The chunk's per-token values, chunk-local angles, and the rotated Bt, Ct
// tiles ([64][N] rows (t, r), TF32-rounded; zero past the sequence end).
// Rt (optional): the rotation table [Q][N/2] of (cos, sin). s_gt: [TG][N/2] scratch.
// bf16 element e of a row of packed pairs, as fp32
__device__ __forceinline__ float bf_word(uint32_t w, int half) {
  return __uint_as_float(half ? (w & 0xffff0000u) : (w << 16));
}

template <int R, int NS, int SB, bool PERM = false>
__device__ __forceinline__ void chunk_prep(const BwdArgs& a, int64_t b, int64_t h, int64_t gi,
                                           int c0, int nv, float A_h, float* Bt, float* Ct,
                                           float2* Rt, TokTab& tk, float* s_gt, float* phi_end) {
  using K = BCfg<R, NS>;
  constexpr int Q = K::Q, K2 = K::K2, TPG = K::TPG;
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t L = a.L, H = a.H, G = a.G;
  // the fold's thread (pair kk, token group tg) takes tokens tg TPG .. + TPG - 1;
  // every global load of the prologue is issued here, before the first barrier
  const int kk = tid % K2, tg = tid / K2;
  float th[TPG];
  uint32_t bw[TPG][R], cw[TPG][R];  // B, C rows 2kk, 2kk + 1 of each token (2R bf16)
  const __nv_bfloat16* Bg = static_cast<const __nv_bfloat16*>(a.B);
  const __nv_bfloat16* Cg = static_cast<const __nv_bfloat16*>(a.C);
#pragma unroll
  for (int j = 0; j < TPG; ++j) {
    const int t = tg * TPG + j;
    th[j] = 0.f;
#pragma unroll
    for (int w = 0; w < R; ++w) bw[j][w] = cw[j][w] = 0u;
    if (t < nv) {
      th[j] = a.theta[((b * L + c0 + t) * G + gi) * K2 + kk];
      const int64_t bc = ((b * L + c0 + t) * G + gi) * NS * R + 2 * kk * R;
      if constexpr (R == 1) {
        bw[j][0] = *reinterpret_cast<const uint32_t*>(Bg + bc);
        cw[j][0] = *reinterpret_cast<const uint32_t*>(Cg + bc);
      } else if constexpr (R == 2) {
        const uint2 u = *reinterpret_cast<const uint2*>(Bg + bc);
        const uint2 v = *reinterpret_cast<const uint2*>(Cg + bc);
        bw[j][0] = u.x; bw[j][1] = u.y;
        cw[j][0] = v.x; cw[j][1] = v.y;
      } else {
        const uint4 u = *reinterpret_cast<const uint4*>(Bg + bc);
        const uint4 v = *reinterpret_cast<const uint4*>(Cg + bc);
        bw[j][0] = u.x; bw[j][1] = u.y; bw[j][2] = u.z; bw[j][3] = u.w;
        cw[j][0] = v.x; cw[j][1] = v.y; cw[j][2] = v.z; cw[j][3] = v.w;
      }
    }
  }
  float bb[2 * R], cb[2 * R];  // the head's biases of rows 2kk, 2kk + 1
#pragma unroll
  for (int e = 0; e < 2 * R; ++e) {
    bb[e] = a.B_bias ? a.B_bias[(h * NS + 2 * kk) * R + e] : 0.f;
    cb[e] = a.C_bias ? a.C_bias[(h * NS + 2 * kk) * R + e] : 0.f;
  }
  if (tid <= Q) {
    const int t = tid;
    float d = 0.f, lm = 0.f;
    if (c0 + t < L && (t < nv || t == Q)) {
      const int64_t o = (b * L + c0 + t) * H + h;
      d = a.dt[o];
      lm = a.lam[o];
    }
    if (t < Q) {
      tk.dt[t] = d;
      tk.lm[t] = lm;
      tk.gam[t] = lm * d;
      tk.lc[t] = d * A_h;
    } else {
      tk.dtn = d;
      tk.lmn = lm;
    }
    tk.bh[t] = (1.f - lm) * d;
  }
  __syncthreads();
  // warp 0: the inclusive sum of dt A over the chunk, then w and e^Lam
  if (tid < 32) {
    float v0 = 2 * lane < Q ? tk.lc[2 * lane] : 0.f;
    float v1 = 2 * lane + 1 < Q ? tk.lc[2 * lane + 1] : 0.f;
    v1 += v0;
    float s = v1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += u;
    }
    const float excl = s - v1;
    const float l0 = excl + v0, l1 = excl + v1;
    const float lend = __shfl_sync(0xffffffffu, s, (Q - 1) / 2);
    if (2 * lane < Q) tk.lc[2 * lane] = l0;
    if (2 * lane + 1 < Q) tk.lc[2 * lane + 1] = l1;
    __syncwarp();
    if (2 * lane < Q) {
      const int t = 2 * lane;
      tk.el[t] = __expf(l0);
      tk.w[t] = __expf(lend - l0) * (tk.gam[t] + tk.bh[t + 1]);
    }
    if (2 * lane + 1 < Q) {
      const int t = 2 * lane + 1;
      tk.el[t] = __expf(l1);
      tk.w[t] = __expf(lend - l1) * (tk.gam[t] + tk.bh[t + 1]);
    }
  }
  // the chunk-local angles: this thread's prefix over its tokens, then the
  // totals of the earlier token groups
  float ang[TPG];
  {
    float run = 0.f;
#pragma unroll
    for (int j = 0; j < TPG; ++j) {
      run += tk.dt[tg * TPG + j] * th[j];
      ang[j] = run;
    }
    s_gt[tg * K2 + kk] = run;
  }
  __syncthreads();
  float off = 0.f;
  for (int q = 0; q < tg; ++q) off += s_gt[q * K2 + kk];
#pragma unroll
  for (int j = 0; j < TPG; ++j) {
    const int t = tg * TPG + j;
    const float phi = off + ang[j];
    if (phi_end && t == Q - 1) phi_end[kk] = phi;
    float sn, cs;
    __sincosf(wrap_angle(phi), &sn, &cs);
    if (Rt) Rt[t * K::RP + kk] = make_float2(cs, sn);
    const bool live = t < nv;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      // elements r (row 2kk) and R + r (row 2kk + 1) of the token's 2R
      const float b0 = live ? bf_word(bw[j][r >> 1], r & 1) + bb[r] : 0.f;
      const float b1 = live ? bf_word(bw[j][(R + r) >> 1], (R + r) & 1) + bb[R + r] : 0.f;
      const float q0 = live ? bf_word(cw[j][r >> 1], r & 1) + cb[r] : 0.f;
      const float q1 = live ? bf_word(cw[j][(R + r) >> 1], (R + r) & 1) + cb[R + r] : 0.f;
      const int row = PERM ? prow(t * R + r) : t * R + r;
      *reinterpret_cast<float2*>(Bt + row * SB + 2 * kk) =
          make_float2(tf32r(cs * b0 + sn * b1), tf32r(cs * b1 - sn * b0));
      *reinterpret_cast<float2*>(Ct + row * SB + 2 * kk) =
          make_float2(tf32r(cs * q0 + sn * q1), tf32r(cs * q1 - sn * q0));
    }
  }
  __syncthreads();
}

// A [64][P] activation tile (rows (t, r), word stride ST) from x-like
// [b,L,H,P,R] bf16, in two halves: each thread's loads of 4 bf16 pairs (a
// warp reads 64 consecutive elements of one token; zero past the sequence
// end), issued early, and their stores, each row scaled by scale[t]; for ST =
// 4 or 8 (mod 32) the stores fill rows without bank conflicts.
template <int R>
__device__ __forceinline__ void act_ld2(uint32_t (&w)[4], const __nv_bfloat16* src, int64_t b,
                                        int64_t h, int64_t L, int64_t H, int c0, int nv) {
  constexpr int PR = kPd * R;
  static_assert(kRows * kPd == 8 * kBT, "four bf16 pairs per thread and tile");
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int e = 2 * (threadIdx.x + k * kBT), t = e / PR, rem = e - t * PR;
    w[k] = t < nv ? *reinterpret_cast<const uint32_t*>(src + ((b * L + c0 + t) * H + h) * PR + rem)
                  : 0u;
  }
}

template <int R, int ST>
__device__ __forceinline__ void act_st2(float* T, const uint32_t (&w)[4], const float* scale) {
  constexpr int PR = kPd * R;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int e = 2 * (threadIdx.x + k * kBT), t = e / PR, rem = e - t * PR;
    const float sc = scale[t];
    const float v0 = tf32r(sc * bf_word(w[k], 0)), v1 = tf32r(sc * bf_word(w[k], 1));
    if (R == 1) {
      *reinterpret_cast<float2*>(T + t * ST + rem) = make_float2(v0, v1);
    } else {
      const int p = rem / R, r = rem % R;
      T[(t * R + r) * ST + p] = v0;
      T[(t * R + r + 1) * ST + p] = v1;
    }
  }
}

// The [64][P] tile of one chunk split in two: each thread's 16-byte load of 8
// consecutive elements of a token (issued early, zero past the sequence end)
// and its stores.
template <int R>
__device__ __forceinline__ uint4 act_ld8(const __nv_bfloat16* src, int64_t b, int64_t h,
                                         int64_t L, int64_t H, int c0, int nv) {
  constexpr int PR = kPd * R;
  const int e = threadIdx.x * 8, t = e / PR, rem = e - t * PR;
  if (t >= nv) return make_uint4(0u, 0u, 0u, 0u);
  return *reinterpret_cast<const uint4*>(src + ((b * L + c0 + t) * H + h) * PR + rem);
}

template <int R, int ST>
__device__ __forceinline__ void act_st8(float* T, uint4 u) {
  constexpr int PR = kPd * R;
  const int e = threadIdx.x * 8, t = e / PR, rem = e - t * PR;
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  if constexpr (R == 1) {
    // 8 consecutive elements of one row: two 16-byte stores (a quarter-warp
    // fills 128 contiguous bytes)
    static_assert(ST % 4 == 0, "16-byte aligned rows");
    float4* d = reinterpret_cast<float4*>(T + prow(t) * ST + rem);
    d[0] = make_float4(bf_word(w[0], 0), bf_word(w[0], 1), bf_word(w[1], 0), bf_word(w[1], 1));
    d[1] = make_float4(bf_word(w[2], 0), bf_word(w[2], 1), bf_word(w[3], 0), bf_word(w[3], 1));
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int p = (rem + i) / R, r = (rem + i) % R;
      T[prow(t * R + r) * ST + p] = bf_word(w[i >> 1], i & 1);
    }
  }
}

// ---------------------------------------------------------------- parts

template <int R, int NS>
constexpr size_t parts_smem() {
  using K = BCfg<R, NS>;
  return sizeof(float) * (2 * kRows * (NS + 8) + 2 * kRows * (kPd + 8) + K::TG * K::K2) +
         sizeof(TokTab);
}

template <int R, int NS>
__global__ void __launch_bounds__(kBT, 2)
    bwd_parts_kernel(BwdArgs a, float* wsA, float* wsB, float* lam_end, float* phi_end, int nC) {
  using K = BCfg<R, NS>;
  constexpr int Q = K::Q, K2 = K::K2;
  // word strides 8 (mod 32): every tile here is read k-major (lanes tq rows
  // apart, g columns apart), which then touches 32 different banks
  constexpr int SBP = NS + 8, SXP = kPd + 8;
  extern __shared__ float4 smf4[];
  float* sm = reinterpret_cast<float*>(smf4);
  float* Bt = sm;
  float* Ct = Bt + kRows * SBP;
  float* Xw = Ct + kRows * SBP;
  float* Ye = Xw + kRows * SXP;
  float* s_gt = Ye + kRows * SXP;
  TokTab& tk = *reinterpret_cast<TokTab*>(s_gt + K::TG * K2);
  const int c = blockIdx.x;
  const int64_t bhi = blockIdx.y, b = bhi / a.H, h = bhi % a.H, gi = h / (a.H / a.G);
  const int c0 = c * Q;
  const int nv = (int)(a.L - c0 < Q ? a.L - c0 : Q);
  const float A_h = a.A[h];
  float* pe = phi_end + (bhi * nC + c) * K2;
  uint32_t xw[4], yw[4];  // x and dy, loaded while the prologue runs
  act_ld2<R>(xw, static_cast<const __nv_bfloat16*>(a.x), b, h, a.L, a.H, c0, nv);
  act_ld2<R>(yw, static_cast<const __nv_bfloat16*>(a.dy), b, h, a.L, a.H, c0, nv);
  chunk_prep<R, NS, SBP>(a, b, h, gi, c0, nv, A_h, Bt, Ct, nullptr, tk, s_gt, pe);
  act_st2<R, SXP>(Xw, xw, tk.w);
  act_st2<R, SXP>(Ye, yw, tk.el);
  if (threadIdx.x == 0) lam_end[bhi * nC + c] = tk.lc[Q - 1];
  __syncthreads();
  // [N][P] = Bt^T Xw and Ct^T Ye: warp tile 16 rows x (8 NT) columns
  constexpr int MT = NS / 16, WPM = 16 / MT, NT = 8 / WPM;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, tq = lane & 3;
  const int m0 = 16 * (warp / WPM), n0 = 8 * NT * (warp % WPM);
  float acc[NT][4];
  const size_t slot = (size_t)(bhi * nC + c) * NS * kPd;
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    zero_acc(acc);
    wgemm_kk<NT, kRows, SBP, SXP>(acc, pass ? Ct : Bt, m0, pass ? Ye : Xw, n0, lane);
    float* dst = (pass ? wsB : wsA) + slot;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int col = n0 + 8 * nt + 2 * tq;
      *reinterpret_cast<float2*>(dst + (m0 + g) * kPd + col) = make_float2(acc[nt][0], acc[nt][1]);
      *reinterpret_cast<float2*>(dst + (m0 + g + 8) * kPd + col) =
          make_float2(acc[nt][2], acc[nt][3]);
    }
  }
}

// ---------------------------------------------------------------- scan

// One thread per (b, h, pair k, column p): the forward recurrence over the
// chunk boundaries (wsA: the parts on entry, H_in of every chunk on exit) and
// the reverse one (wsB: the parts on entry, dG of every chunk on exit), with
// the chunk-end rotation's angle gradient (dphiB) and <dG, H_in> (dotgh).
template <int NS>
__global__ void __launch_bounds__(256)
    bwd_scan_kernel(const float* __restrict__ lam_end, const float* __restrict__ phi_end,
                    float* __restrict__ wsA, float* __restrict__ wsB,
                    const float* __restrict__ d_final, float* __restrict__ dphiB,
                    float* __restrict__ dotgh, int nC) {
  constexpr int K2 = NS / 2;
  constexpr int kB = 8;  // chunks whose loads are issued together
  const int64_t bhi = blockIdx.x;
  const int k = blockIdx.y * 4 + (int)(threadIdx.x >> 6), p = threadIdx.x & 63;
  const int lane = threadIdx.x & 31;
  const float* le = lam_end + bhi * nC;
  const float* pe = phi_end + bhi * nC * K2 + k;
  float* A0 = wsA + (size_t)bhi * nC * NS * kPd + (2 * k) * kPd + p;
  float* B0 = wsB + (size_t)bhi * nC * NS * kPd + (2 * k) * kPd + p;
  constexpr size_t kSlot = (size_t)NS * kPd;
  float h0 = 0.f, h1 = 0.f;
  for (int c1 = 0; c1 < nC; c1 += kB) {
    const int n = nC - c1 < kB ? nC - c1 : kB;
    float g0[kB], g1[kB], e[kB], ph[kB];
#pragma unroll
    for (int j = 0; j < kB; ++j)
      if (j < n) {
        const float* q = A0 + (c1 + j) * kSlot;
        g0[j] = q[0];
        g1[j] = q[kPd];
        e[j] = le[c1 + j];
        ph[j] = pe[(c1 + j) * K2];
      }
#pragma unroll
    for (int j = 0; j < kB; ++j)
      if (j < n) {
        float* q = A0 + (c1 + j) * kSlot;
        q[0] = h0;
        q[kPd] = h1;
        float sn, cs;
        __sincosf(wrap_angle(ph[j]), &sn, &cs);
        const float ee = __expf(e[j]);
        const float G0 = fmaf(ee, h0, g0[j]), G1 = fmaf(ee, h1, g1[j]);
        h0 = cs * G0 - sn * G1;
        h1 = sn * G0 + cs * G1;
      }
  }
  float dh0 = 0.f, dh1 = 0.f;
  if (d_final) {
    const float* df = d_final + (size_t)bhi * NS * kPd + (2 * k) * kPd + p;
    dh0 = df[0];
    dh1 = df[kPd];
  }
  float o0 = h0, o1 = h1;  // the state leaving chunk c
  for (int c1 = nC - 1; c1 >= 0; c1 -= kB) {
    const int n = c1 + 1 < kB ? c1 + 1 : kB;  // chunks c1, c1 - 1, .., c1 - n + 1
    float i0[kB], i1[kB], d0[kB], d1[kB], e[kB], ph[kB];
#pragma unroll
    for (int j = 0; j < kB; ++j)
      if (j < n) {
        const int c = c1 - j;
        i0[j] = A0[c * kSlot];
        i1[j] = A0[c * kSlot + kPd];
        d0[j] = B0[c * kSlot];
        d1[j] = B0[c * kSlot + kPd];
        e[j] = le[c];
        ph[j] = pe[c * K2];
      }
#pragma unroll
    for (int j = 0; j < kB; ++j)
      if (j < n) {
        const int c = c1 - j;
        float sn, cs;
        __sincosf(wrap_angle(ph[j]), &sn, &cs);
        const float dg0 = cs * dh0 + sn * dh1, dg1 = cs * dh1 - sn * dh0;
        float dp = dh1 * o0 - dh0 * o1;
        float dot = dg0 * i0[j] + dg1 * i1[j];
        B0[c * kSlot] = dg0;
        B0[c * kSlot + kPd] = dg1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          dp += __shfl_xor_sync(0xffffffffu, dp, o);
          dot += __shfl_xor_sync(0xffffffffu, dot, o);
        }
        if (lane == 0) {
          atomicAdd(dphiB + (bhi * nC + c) * K2 + k, dp);
          atomicAdd(dotgh + bhi * nC + c, dot);
        }
        const float ee = __expf(e[j]);
        dh0 = fmaf(ee, dg0, d0[j]);
        dh1 = fmaf(ee, dg1, d1[j]);
        o0 = i0[j];
        o1 = i1[j];
      }
  }
}

// ---------------------------------------------------------------- chunk

template <int R, int NS>
constexpr size_t chunk_smem() {
  using K = BCfg<R, NS>;
  return sizeof(float) * (2 * kRows * K::SB + 5 * kRows * kSX + NS * kSX + 2 * K::Q * K::RP +
                          K::TG * K::K2 + 8 * kRows) +
         sizeof(TokTab);
}

template <int R, int NS>
__global__ void __launch_bounds__(kBT, 1)
    bwd_chunk_kernel(BwdArgs a, const float* wsA, const float* wsB, const float* dphiB,
                     const float* dotgh, int nC) {
  using K = BCfg<R, NS>;
  constexpr int Q = K::Q, K2 = K::K2, SB = K::SB;
  extern __shared__ float4 smf4[];
  float* sm = reinterpret_cast<float*>(smf4);
  float* Bt = sm;
  float* Ct = Bt + kRows * SB;
  float* Xs = Ct + kRows * SB;
  float* Ys = Xs + kRows * kSX;
  float* PT = Ys + kRows * kSX;   // P transposed: [s row][t row]
  float* dSs = PT + kRows * kSX;  // dS
  float* dST = dSs + kRows * kSX; // dS transposed
  float* St = dST + kRows * kSX;  // [N][P]: H_in, then dG
  float2* Rt = reinterpret_cast<float2*>(St + NS * kSX);  // [Q][RP] (cos, sin) of the angles
  // [Q][K2] angle gradients (row pitch K2 + 4: the stores of a warp's 8 rows
  // x 4 pairs fall on different banks), once X is no longer read
  constexpr int kDP = K2 + 4;
  static_assert(Q * kDP <= kRows * kSX, "the angle gradients fit the X tile");
  float* dPh = Xs;
  float* s_gt = reinterpret_cast<float*>(Rt + Q * K::RP);
  float* colVi = s_gt + K::TG * K2;  // per token: column sums and row sums (64 each)
  float* colVs = colVi + kRows;
  float* colZ = colVs + kRows;
  float* rowZ = colZ + kRows;
  float* elg = rowZ + kRows;
  float* dwv = elg + kRows;
  float* ths = dwv + kRows;
  float* dlv = ths + kRows;
  TokTab& tk = *reinterpret_cast<TokTab*>(dlv + kRows);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tq = lane & 3;
  const int c = blockIdx.x;
  const int64_t bhi = blockIdx.y, b = bhi / a.H, h = bhi % a.H, gi = h / (a.H / a.G);
  const int64_t L = a.L, H = a.H, G = a.G;
  const int c0 = c * Q;
  const int nv = (int)(L - c0 < Q ? L - c0 : Q);
  const float A_h = a.A[h];
  const size_t slot = (size_t)(bhi * nC + c) * NS * kPd;
  const uint32_t aBt = ptx::smem_addr(Bt), aCt = ptx::smem_addr(Ct), aXs = ptx::smem_addr(Xs),
                 aYs = ptx::smem_addr(Ys), aPT = ptx::smem_addr(PT), adS = ptx::smem_addr(dSs),
                 adST = ptx::smem_addr(dST), aSt = ptx::smem_addr(St);

  // the chunk's x, dy and entering state, loaded into registers while the
  // prologue runs (one 64 x 64 tile is exactly one 16-byte load per thread)
  static_assert(kRows * kPd == 8 * kBT, "one 16-byte load per thread and tile");
  constexpr int NH = NS * kPd / (4 * kBT);
  const uint4 xr = act_ld8<R>(static_cast<const __nv_bfloat16*>(a.x), b, h, L, H, c0, nv);
  const uint4 yr = act_ld8<R>(static_cast<const __nv_bfloat16*>(a.dy), b, h, L, H, c0, nv);
  float4 hr[NH];
#pragma unroll
  for (int j = 0; j < NH; ++j)
    hr[j] = *reinterpret_cast<const float4*>(wsA + slot + 4 * (tid + j * kBT));
  for (int i = tid; i < 8 * kRows; i += kBT) colVi[i] = 0.f;
  chunk_prep<R, NS, SB, true>(a, b, h, gi, c0, nv, A_h, Bt, Ct, Rt, tk, s_gt, nullptr);
  act_st8<R, kSX>(Xs, xr);
  act_st8<R, kSX>(Ys, yr);
#pragma unroll
  for (int j = 0; j < NH; ++j) {
    const int e = 4 * (tid + j * kBT), n = e / kPd, p = e - n * kPd;
    *reinterpret_cast<float4*>(St + prow(n) * kSX + p) =
        make_float4(tf32r(hr[j].x), tf32r(hr[j].y), tf32r(hr[j].z), tf32r(hr[j].w));
  }
  __syncthreads();

  // ---- S = Ct Bt^T, dP = dY X^T (64 x 64; warp tile 16 x 16), the masks
  {
    const int m0 = 16 * (warp >> 2), n0 = 16 * (warp & 3);
    float aS[2][4], aP[2][4];
    zero_acc(aS);
    zero_acc(aP);
    wgemm_l<2, NS, SB, SB, true, true>(aS, aCt, m0, aBt, nullptr, n0, lane);
    wgemm_l<2, kPd, kSX, kSX, true, true>(aP, aYs, m0, aXs, nullptr, n0, lane);
    float rz[2] = {0.f, 0.f};
    float cvi[2][2], cvs[2][2], cz[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int q = 0; q < 2; ++q) cvi[nt][q] = cvs[nt][q] = cz[nt][q] = 0.f;
    // the token values of the thread's two rows and four columns
    float lr[2], lcol[2][2], gcol[2][2], bcol[2][2];
#pragma unroll
    for (int q = 0; q < 2; ++q) lr[q] = tk.lc[(m0 + g + 8 * q) / R];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int s = (n0 + 8 * nt + 2 * tq + q) / R;
        lcol[nt][q] = tk.lc[s];
        gcol[nt][q] = tk.gam[s];
        bcol[nt][q] = tk.bh[s + 1];
      }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = m0 + g + 8 * (e >> 1), j = n0 + 8 * nt + 2 * tq + (e & 1);
        const int t = i / R, s = j / R;
        float pv = 0.f, dsv = 0.f;
        if (t >= s) {
          const float D = __expf(lr[e >> 1] - lcol[nt][e & 1]);
          const float f = gcol[nt][e & 1] + (s < t ? bcol[nt][e & 1] : 0.f);
          const float M = D * f;
          pv = aS[nt][e] * M;
          dsv = aP[nt][e] * M;
          const float sd = aS[nt][e] * aP[nt][e] * D;
          cvi[nt][e & 1] += sd;
          if (s < t) {
            const float z = sd * f;
            cvs[nt][e & 1] += sd;
            cz[nt][e & 1] += z;
            rz[e >> 1] += z;
          }
        }
        PT[j * kSX + i] = tf32r(pv);
        dSs[i * kSX + j] = tf32r(dsv);
        dST[j * kSX + i] = tf32r(dsv);
      }
    // column sums over the warp's 16 rows (lanes that differ in g)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int q = 0; q < 2; ++q) {
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          cvi[nt][q] += __shfl_xor_sync(0xffffffffu, cvi[nt][q], o);
          cvs[nt][q] += __shfl_xor_sync(0xffffffffu, cvs[nt][q], o);
          cz[nt][q] += __shfl_xor_sync(0xffffffffu, cz[nt][q], o);
        }
        if (g == 0) {
          const int s = (n0 + 8 * nt + 2 * tq + q) / R;
          atomicAdd(&colVi[s], cvi[nt][q]);
          atomicAdd(&colVs[s], cvs[nt][q]);
          atomicAdd(&colZ[s], cz[nt][q]);
        }
      }
    // row sums over the warp's 16 columns (lanes that differ in tq)
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      rz[q] += __shfl_xor_sync(0xffffffffu, rz[q], 1);
      rz[q] += __shfl_xor_sync(0xffffffffu, rz[q], 2);
      if (tq == 0) atomicAdd(&rowZ[(m0 + g + 8 * q) / R], rz[q]);
    }
  }
  __syncthreads();

  // ---- dCt = diag(e^Lam) dY H_in^T + dS Bt, and dBt = diag(w) X dG^T + dS^T Ct
  //      (64 x N; warp tile 16 x N/4), each followed by the rotation backward
  constexpr int NT3 = NS / 32;
  const int m0 = 16 * (warp >> 2), n0 = (NS / 4) * (warp & 3);
  float dphr[2][NT3];  // the angle gradient of (row m0 + g + 8q, pair of n-tile nt)
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int nt = 0; nt < NT3; ++nt) dphr[q][nt] = 0.f;
  float4 gr[NH];  // dG, loaded during the first pass
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    if (pass == 1) {
      // the state tile: H_in -> dG
      __syncthreads();
#pragma unroll
      for (int j = 0; j < NH; ++j) {
        const int e = 4 * (tid + j * kBT), n = e / kPd, p = e - n * kPd;
        *reinterpret_cast<float4*>(St + prow(n) * kSX + p) =
            make_float4(tf32r(gr[j].x), tf32r(gr[j].y), tf32r(gr[j].z), tf32r(gr[j].w));
      }
      __syncthreads();
    }
    const float* Own = pass ? Bt : Ct;   // the tile whose gradient this is
    const float* Oth = pass ? Ct : Bt;   // the other factor of S
    float acc[NT3][4];
    zero_acc(acc);
    // E = (pass 0) dY H_in^T, (pass 1) X dG^T
    wgemm_l<NT3, kPd, kSX, kSX, true, true>(acc, pass ? aXs : aYs, m0, aSt, nullptr, n0, lane);
    // row dots with the own tile: d e^Lam_t (pass 0), dw_s (pass 1)
    {
      float rd[2] = {0.f, 0.f};
#pragma unroll
      for (int nt = 0; nt < NT3; ++nt) {
        const int col = n0 + 8 * nt + 2 * tq;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const float2 o = *reinterpret_cast<const float2*>(Own + prow(m0 + g + 8 * q) * SB + col);
          rd[q] = fmaf(o.x, acc[nt][2 * q], fmaf(o.y, acc[nt][2 * q + 1], rd[q]));
        }
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        rd[q] += __shfl_xor_sync(0xffffffffu, rd[q], 1);
        rd[q] += __shfl_xor_sync(0xffffffffu, rd[q], 2);
        if (tq == 0) atomicAdd(&(pass ? dwv : elg)[(m0 + g + 8 * q) / R], rd[q]);
      }
    }
    // scale the rows: e^Lam_t (pass 0), w_s (pass 1)
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int t = (m0 + g + 8 * q) / R;
      const float sc = pass ? tk.w[t] : tk.el[t];
#pragma unroll
      for (int nt = 0; nt < NT3; ++nt) {
        acc[nt][2 * q] *= sc;
        acc[nt][2 * q + 1] *= sc;
      }
    }
    // + dS Oth (pass 0) or dS^T Oth (pass 1)
    wgemm_l<NT3, kRows, kSX, SB, false, false>(acc, pass ? adST : adS, m0, 0u, Oth, n0, lane);
    if (pass == 0) {
#pragma unroll
      for (int j = 0; j < NH; ++j)
        gr[j] = *reinterpret_cast<const float4*>(wsB + slot + 4 * (tid + j * kBT));
    }
    // rotation backward: the raw gradient Rot(Phi_t) d, the angle gradient,
    // and the bias gradient (summed over the warp's rows of equal rank)
    float* graw = pass ? a.dB : a.dC;
    float* gbias = pass ? a.dB_bias : a.dC_bias;
    float* grow[2];  // the raw gradient's row of each of the thread's two rows
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int i = m0 + g + 8 * q, t = i / R, r = i % R;
      grow[q] = graw + ((b * L + c0 + t) * G + gi) * NS * R + r;
    }
#pragma unroll
    for (int nt = 0; nt < NT3; ++nt) {
      const int col = n0 + 8 * nt + 2 * tq, k = col >> 1;
      float bs0 = 0.f, bs1 = 0.f;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int i = m0 + g + 8 * q, t = i / R;
        const float d0 = acc[nt][2 * q], d1 = acc[nt][2 * q + 1];
        const float2 o = *reinterpret_cast<const float2*>(Own + prow(i) * SB + col);
        dphr[q][nt] += d0 * o.y - d1 * o.x;
        const float2 rt = Rt[t * K::RP + k];
        const float r0 = rt.x * d0 - rt.y * d1, r1 = rt.y * d0 + rt.x * d1;
        if (t < nv) {
          float* dst = grow[q] + col * R;
          if (R == 1) {
            atomicAdd(reinterpret_cast<float2*>(dst), make_float2(r0, r1));
          } else {
            atomicAdd(dst, r0);
            atomicAdd(dst + R, r1);
          }
        }
        bs0 += r0;
        bs1 += r1;
      }
      if (gbias) {
        // rows m0 + g and m0 + g + 8 have rank g % R: sum over the lanes of equal rank
#pragma unroll
        for (int o = 4 * R; o < 32; o <<= 1) {
          bs0 += __shfl_xor_sync(0xffffffffu, bs0, o);
          bs1 += __shfl_xor_sync(0xffffffffu, bs1, o);
        }
        if (g < R) {
          atomicAdd(gbias + (h * NS + col) * R + g, bs0);
          atomicAdd(gbias + (h * NS + col + 1) * R + g, bs1);
        }
      }
    }
  }

  // theta of the angle pass below (thread (pair, token group) as in the fold),
  // loaded while dX is formed
  constexpr int TG = K::TG, TPG = K::TPG;
  float thv[TPG];
  {
    const int kk = tid % K2, tg = tid / K2;
#pragma unroll
    for (int j = 0; j < TPG; ++j) {
      const int t = tg * TPG + j;
      thv[j] = t < nv ? a.theta[((b * L + c0 + t) * G + gi) * K2 + kk] : 0.f;
    }
  }
  // ---- dX = P^T dY + diag(w) Bt dG (64 x 64; warp tile 16 x 16)
  {
    const int xm0 = 16 * (warp >> 2), xn0 = 16 * (warp & 3);
    float a1[2][4], a2[2][4];
    zero_acc(a1);
    zero_acc(a2);
    wgemm_l<2, kRows, kSX, kSX, false, false>(a1, aPT, xm0, 0u, Ys, xn0, lane);
    wgemm_l<2, NS, SB, kSX, false, true>(a2, aBt, xm0, 0u, St, xn0, lane);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int j = xm0 + g + 8 * q, s = j / R, r = j % R;
      if (s >= nv) continue;
      const float ws = tk.w[s];
      float* dst = a.dx + ((b * L + c0 + s) * H + h) * kPd * R + r;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int p = xn0 + 8 * nt + 2 * tq;
        dst[p * R] = fmaf(ws, a2[nt][2 * q], a1[nt][2 * q]);
        dst[(p + 1) * R] = fmaf(ws, a2[nt][2 * q + 1], a1[nt][2 * q + 1]);
      }
    }
  }
  __syncthreads();
  // the angle gradients of the rows into dPh (X is no longer read); rows of
  // one token (R > 1) are summed over the lanes that hold them
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int nt = 0; nt < NT3; ++nt) {
      float v = dphr[q][nt];
      if (R >= 2) v += __shfl_xor_sync(0xffffffffu, v, 4);
      if (R >= 4) v += __shfl_xor_sync(0xffffffffu, v, 8);
      const int i = m0 + g + 8 * q, k = (n0 + 8 * nt + 2 * tq) >> 1;
      if (g % R == 0) dPh[(i / R) * kDP + k] = v;
    }
  __syncthreads();

  // ---- the angle gradients: the chunk-end rotation at the last token, the
  //      reverse sum over the chunk's tokens, dtheta, and theta . dphi per
  //      token; thread (pair kk, token group tg) as in the fold
  {
    const int kk = tid % K2, tg = tid / K2;
    float run[TPG];
    float acc = (tg == TG - 1) ? dphiB[(bhi * nC + c) * K2 + kk] : 0.f;
#pragma unroll
    for (int j = TPG - 1; j >= 0; --j) {
      const int t = tg * TPG + j;
      acc += dPh[t * kDP + kk];
      run[j] = acc;
    }
    s_gt[tg * K2 + kk] = acc;
    __syncthreads();
    float off = 0.f;
    for (int q = tg + 1; q < TG; ++q) off += s_gt[q * K2 + kk];
#pragma unroll
    for (int j = 0; j < TPG; ++j) {
      const int t = tg * TPG + j;
      const float dphi = off + run[j];
      if (t < nv) atomicAdd(a.dtheta + ((b * L + c0 + t) * G + gi) * K2 + kk, tk.dt[t] * dphi);
      // theta . dphi over the pairs: a warp holds 32 pairs of one token
      float v = thv[j] * dphi;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) atomicAdd(&ths[t], v);
    }
  }
  __syncthreads();

  // ---- decay and trapezoid gradients per token (warp 0, two tokens a lane)
  if (warp == 0) {
    const float lend = tk.lc[Q - 1];
    const float eend = __expf(lend) * dotgh[bhi * nC + c];
    float fz[2], fe[2], fw[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int u = 2 * lane + q;
      fz[q] = u < Q ? colZ[u] - rowZ[u] : 0.f;
      fe[q] = u < Q ? elg[u] * tk.el[u] : 0.f;
      fw[q] = u < Q ? dwv[u] * tk.w[u] : 0.f;
    }
    // exclusive prefix of fz and fw, inclusive suffix of fe (over u = 2 lane + q)
    float pz = fz[0] + fz[1], pw = fw[0] + fw[1], se = fe[0] + fe[1];
    float iz = pz, iw = pw, is = se;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float uz = __shfl_up_sync(0xffffffffu, iz, o);
      const float uw = __shfl_up_sync(0xffffffffu, iw, o);
      const float us = __shfl_down_sync(0xffffffffu, is, o);
      if (lane >= o) {
        iz += uz;
        iw += uw;
      }
      if (lane + o < 32) is += us;
    }
    const float ez = iz - pz, ew = iw - pw;  // sums over u' < 2 lane
    const float es = is - se;                // sum over u' > 2 lane + 1
    float dA_part = 0.f;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int u = 2 * lane + q;
      const float F = ez + (q ? fz[0] : 0.f);
      const float Sw = ew + (q ? fw[0] : 0.f);
      const float Se = es + fe[1] + (q ? 0.f : fe[0]);
      if (u < nv) {
        const float dl = F + Se + Sw + eend;
        const float dgam = colVi[u] + dwv[u] * __expf(lend - tk.lc[u]);
        const float dbh = u >= 1 ? colVs[u - 1] + dwv[u - 1] * __expf(lend - tk.lc[u - 1]) : 0.f;
        const float d = tk.dt[u], lm = tk.lm[u];
        const int64_t o = (b * L + c0 + u) * H + h;
        atomicAdd(a.ddt + o, A_h * dl + lm * dgam + (1.f - lm) * dbh + ths[u]);
        atomicAdd(a.dlam + o, d * (dgam - dbh));
        dA_part = fmaf(d, dl, dA_part);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dA_part += __shfl_xor_sync(0xffffffffu, dA_part, o);
    if (lane == 0) {
      atomicAdd(a.dA + h, dA_part);
      // the trapezoid weight of the token after the chunk enters this chunk's w
      if (c0 + Q < L) {
        const float dbn = dwv[Q - 1];
        const int64_t o = (b * L + c0 + Q) * H + h;
        atomicAdd(a.ddt + o, (1.f - tk.lmn) * dbn);
        atomicAdd(a.dlam + o, -tk.dtn * dbn);
      }
    }
  }
}

template <int R, int NS>
cudaError_t launch_rn(const BwdArgs& a, float* ws, int nC, cudaStream_t s) {
  constexpr int K2 = NS / 2;
  const int64_t nbh = a.batch * a.H;
  const size_t big = (size_t)nbh * nC * NS * kPd;
  float* wsA = ws;
  float* wsB = wsA + big;
  float* lam_end = wsB + big;
  float* phi_end = lam_end + (size_t)nbh * nC;
  float* dphiB = phi_end + (size_t)nbh * nC * K2;
  float* dotgh = dphiB + (size_t)nbh * nC * K2;
  cudaError_t e = cudaMemsetAsync(dphiB, 0, sizeof(float) * (size_t)nbh * nC * (K2 + 1), s);
  if (e != cudaSuccess) return e;
  static_assert(chunk_smem<R, NS>() <= 227 * 1024 && parts_smem<R, NS>() <= 227 * 1024,
                "the per-chunk tiles fit one CTA's shared memory");
  const size_t sp = parts_smem<R, NS>(), sc = chunk_smem<R, NS>();
  e = cudaFuncSetAttribute(bwd_parts_kernel<R, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)sp);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(bwd_chunk_kernel<R, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)sc);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)nC, (unsigned)nbh);
  bwd_parts_kernel<R, NS><<<grid, kBT, sp, s>>>(a, wsA, wsB, lam_end, phi_end, nC);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  bwd_scan_kernel<NS><<<dim3((unsigned)nbh, (unsigned)(K2 / 4)), 256, 0, s>>>(
      lam_end, phi_end, wsA, wsB, a.d_final, dphiB, dotgh, nC);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  bwd_chunk_kernel<R, NS><<<grid, kBT, sc, s>>>(a, wsA, wsB, dphiB, dotgh, nC);
  return cudaGetLastError();
}

}  // namespace

bool scan_bwd_tc_ok(const BwdArgs& a, bool bf16) {
  auto al = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!bf16 || a.P != kPd || !(a.N == 64 || a.N == 128)) return false;
  if (!(a.R == 1 || a.R == 2 || a.R == 4)) return false;
  if (a.batch * a.H > 65535) return false;  // grid y
  const int64_t Q = kRows / a.R, nC = (a.L + Q - 1) / Q;
  if (nC > 0x7fffffffLL) return false;
  // 16-byte vectors of x / dy rows and of B / C pairs, 8-byte atomics of dB / dC at R = 1
  if (!al(a.x) || !al(a.dy) || !al(a.B) || !al(a.C) || !al(a.dB) || !al(a.dC)) return false;
  return true;
}

size_t scan_bwd_tc_workspace(const BwdArgs& a) {
  const int64_t Q = kRows / a.R, nC = (a.L + Q - 1) / Q, nbh = a.batch * a.H;
  return sizeof(float) * ((size_t)nbh * nC * (2 * a.N * kPd + 1 + a.N + 1));
}

cudaError_t launch_scan_bwd_tc(const BwdArgs& a, float* ws, cudaStream_t s) {
  const int nC = (int)((a.L + kRows / a.R - 1) / (kRows / a.R));
  switch (a.R * 1000 + (int)a.N) {
    case 1064: return launch_rn<1, 64>(a, ws, nC, s);
    case 1128: return launch_rn<1, 128>(a, ws, nC, s);
    case 2064: return launch_rn<2, 64>(a, ws, nC, s);
    case 2128: return launch_rn<2, 128>(a, ws, nC, s);
    case 4064: return launch_rn<4, 64>(a, ws, nC, s);
    case 4128: return launch_rn<4, 128>(a, ws, nC, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace m3
