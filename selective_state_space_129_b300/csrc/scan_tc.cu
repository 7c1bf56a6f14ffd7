// Tensor-core (tcgen05 + TMEM + TMA) chunked prefill of the Mamba-3 scan.
//
// Scope: bf16 activations, head dim P = 64, state N in {64, 128}, MIMO rank
// R in {1, 2, 4} with chunk Q = 64 / R, so that the flattened (token, rank)
// tile of a chunk has QR = 64 rows (the MIMO chunk rule C_MIMO = C_SISO / R of
// papernotes.org sec. 3).
//
// Math (per batch row b and head h). The rotation of the complex-valued state
// is folded into B and C as a cumulative data-dependent RoPE (aipaper.cc
// sec. 4.2, Prop. 3): with Phi_t = sum_{u<=t} Delta_u theta_u (per state pair,
// over the whole sequence) and Rot(-Phi_t) applied to B_t and C_t,
//   g_t = alpha_t g_{t-1} + beta_t Bt_{t-1} x_{t-1}^T + gamma_t Bt_t x_t^T,
//   y_t = Ct_t^T g_t,   h_t = Rot(Phi_t) g_t   (explicit frame).
// The exponential-trapezoidal weights are those of Prop. 1 (aipaper.cc
// sec. 4.1). The state g therefore needs no rotation between chunks. Within a
// chunk of tokens t0..t1 (Lam = chunk-local inclusive cumsum of Delta A):
//   S   = Ct Bt^T                                   (tcgen05, M=64 N=64 K=N)
//   P   = S o Mask,  Mask[t,s] = exp(Lam_t - Lam_s)(gamma_s + [s<t] bhat_{s+1}),
//         s <= t  -- decay (1-semiseparable) times the 2-band trapezoid mask
//         (papernotes.org sec. 1; SSD form Y = (L o C B^T) X)
//   Y   = P X + diag(exp(Lam_t)) Ct H_in            (two tcgen05 GEMMs)
//   H_out = exp(Lam_t1) H_in + Bt^T diag(w) X,  w_s = exp(Lam_t1 - Lam_s)(gamma_s + bhat_{s+1})
// where H_in is the chunk's entering state including the pending beta term of
// its first token, and bhat_{s+1} = (1 - lambda_{s+1}) Delta_{s+1} (0 past the
// end). H lives in fp32 registers.
//
// Precision. The rotated operands are data derived in fp32, not inputs, and
// the score matrix sums products much larger than y itself (|B|^2 = N for
// RMS-normalised B). Their operand tiles (Bt, Ct, w X and the state copy) are
// therefore fp16 (11-bit significand, kind::f16 MMA with fp32 accumulation),
// each scaled by a power of two chosen per chunk from a block-wide bound of
// its magnitude, so fp16's range never limits the inputs. The scales are undone
// exactly where a per-element factor is applied anyway (mask, state update,
// output). P is split into bf16 high and low parts so that P X (X is an exact
// bf16 input) keeps ~16 significant bits.
//
// One CTA (256 threads, two CTAs per SM) walks one (b, h) sequence chunk by
// chunk. Per chunk:
//   phase 0  warp 0: decay scan, trapezoid weights (warp shuffles)
//   phase 1  all: cumulative angles (per-thread prefix + cross-thread carry),
//            sincos, rotate B/C (+bias) into fp16 UMMA tiles; build w X
//   phase 2  one thread: S, D = Bt^T (w X), Yoff = Ct H_in    (tcgen05.mma)
//   phase 3  all: mask S -> P (bf16 hi + lo); H = exp(Lam_end) H + D
//   phase 4  one thread: Y = P X                               (tcgen05.mma)
//   phase 5  all: y = Y + exp(Lam_t) Yoff -> bf16 -> TMA store; fp16 state copy
// Operand tiles are 128-byte-swizzled rows of 64 16-bit elements; a
// [rows][64k] tile is at once the K-major operand along its columns and the
// MN-major operand along its rows, so Bt serves both S (K = N) and the state
// GEMM (K = tokens).
// Every mbarrier wait is bounded; on expiry the CTA records the status word,
// stops issuing work and still frees its tensor memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace m3 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kQR = 64;  // rows of the flattened (token, rank) tile
constexpr int kP = 64;   // head dim of the tensor-core path
constexpr uint32_t kTmemCols = 256;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s per wait
constexpr uint32_t kTileBytes = 64 * 128;    // 64 rows x 128 B
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kInvTwoPi = 0.15915494309189535f;
// 2 pi = kPi2a + kPi2b + kPi2c (Cody and Waite's additive split): kPi2a has 8
// significant bits, so k * kPi2a is exact for the multiples k used here.
constexpr float kPi2a = 6.28125f;
constexpr float kPi2b = 1.9353071795864769e-3f;
constexpr float kPi2c = 1.0253131677e-11f;

// TMEM column offsets of the four fp32 accumulators.
constexpr uint32_t kColS = 0, kColD = 64, kColY = 128, kColYo = 192;

template <int R, int NS>
struct Cfg {
  static constexpr int Q = kQR / R;         // tokens per chunk
  static constexpr int KP = NS / 2;         // rotating state pairs
  static constexpr int TG = kThreads / KP;  // token groups in the angle phase
  static constexpr int TPG = Q / TG;        // tokens per thread in the angle phase
  static_assert(Q % TG == 0, "token groups must divide the chunk");
  static constexpr int HR = NS * kP / kThreads;  // fp32 state values per thread
  // byte offsets in dynamic shared memory (1024-aligned base)
  static constexpr uint32_t kBt = 0;                          // [64][NS] fp16
  static constexpr uint32_t kCt = kBt + 64 * NS * 2;          // [64][NS] fp16
  static constexpr uint32_t kXs = kCt + 64 * NS * 2;          // 2 TMA stages of x
  static constexpr uint32_t kXb = kXs + 2 * kTileBytes;       // X re-laid (R > 1), bf16
  static constexpr uint32_t kXw = kXb + kTileBytes;           // w-scaled X, fp16
  static constexpr uint32_t kPh = kXw + kTileBytes;           // masked scores, bf16 high
  static constexpr uint32_t kPl = kPh + kTileBytes;           // masked scores, bf16 low
  static constexpr uint32_t kH = kPl + kTileBytes;            // [NS][64] fp16 state copy
  static constexpr uint32_t kYs = kH + NS * 128;              // output staging
  static constexpr uint32_t kBytes = kYs + kTileBytes;
  static constexpr uint32_t kSmem = kBytes + 1024;            // + alignment slack
};

struct TcParams {
  const float* dt;
  const float* A;
  const float* lam;
  const __nv_bfloat16* B;
  const __nv_bfloat16* C;
  const float* theta;
  const float* B_bias;
  const float* C_bias;
  float* final_state;
  unsigned int* status;
  int64_t L, H, G;
  int nchunks;
};

__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t col) {
  return row * 128u + ((((col >> 3) ^ row) & 7u) << 4) + (col & 7u) * 2u;
}
// [rows][K] tile stored as K/64 blocks of [rows][64]: byte offset of (row, col).
__device__ __forceinline__ uint32_t tile_off(uint32_t row, uint32_t col, uint32_t rows) {
  return (col >> 6) * rows * 128u + sw128(row, col & 63u);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
// Largest magnitude of the two bf16 values of a word, as a float.
__device__ __forceinline__ float bf_absmax(uint32_t w) {
  const uint32_t a = w & 0x7fff7fffu;
  return fmaxf(__uint_as_float(a << 16), __uint_as_float(a & 0xffff0000u));
}

// Power of two sigma with M * sigma < 2^15 (inside fp16's range), and 1/sigma.
__device__ __forceinline__ void pow2_scale(float M, float* sigma, float* inv) {
  int e = (int)((__float_as_uint(M) >> 23) & 0xffu) - 127;  // M in [2^e, 2^(e+1))
  e = e < -100 ? -100 : (e > 127 ? 127 : e);
  *sigma = __uint_as_float((uint32_t)(127 + 14 - e) << 23);
  *inv = __uint_as_float((uint32_t)(127 - 14 + e) << 23);
}

// Float-float addition (Knuth's TwoSum, then a renormalising Fast2Sum):
// (ah, al) += (bh, bl) with ~44 significant bits.
__device__ __forceinline__ void ff_add(float& ah, float& al, float bh, float bl) {
  const float s = ah + bh;
  const float v = s - ah;
  float e = (ah - (s - v)) + (bh - v);
  e += al + bl;
  ah = s + e;
  al = e - (ah - s);
}
// Reduce a float-float angle (radians) by the nearest multiple of 2 pi.
__device__ __forceinline__ void ff_wrap(float& ah, float& al) {
  const float k = rintf(ah * kInvTwoPi);
  const float h = fmaf(-k, kPi2a, ah);  // exact: Sterbenz / 8-bit kPi2a
  float l = fmaf(-k, kPi2b, al);
  l = fmaf(-k, kPi2c, l);
  ah = h + l;
  al = l - (ah - h);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void sts64(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void sts16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Shared-memory operand descriptors of the 128-byte-swizzled tiles.
// K-major: 16-element K step kk of a [rows][K] tile.
__device__ __forceinline__ uint64_t desc_k(uint32_t base, int kk, uint32_t rows) {
  return ptx::smem_desc_sw128(base + (uint32_t)(kk >> 2) * rows * 128u + (uint32_t)(kk & 3) * 32u,
                              16u, 1024u);
}
// MN-major: 16-row K step kk of a [K][MN] tile whose 64-wide MN blocks are
// `lbo` bytes apart.
__device__ __forceinline__ uint64_t desc_mn(uint32_t base, int kk, uint32_t lbo) {
  return ptx::smem_desc_sw128(base + (uint32_t)kk * 2048u, lbo, 1024u);
}

// Wait on an mbarrier phase; on expiry record the status word and the CTA's
// abort flag. Returns false once the CTA is aborting.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, int* abort_flag,
                                              unsigned int* status) {
  if (*reinterpret_cast<volatile int*>(abort_flag)) return false;
  if (ptx::mbar_wait(bar, parity, kWaitNs)) return true;
  atomicOr(status, 1u);
  *reinterpret_cast<volatile int*>(abort_flag) = 1;
  return false;
}

template <int R, int NS>
__global__ void __launch_bounds__(kThreads, 2)
    scan_tc_kernel(const __grid_constant__ CUtensorMap tm_x,
                   const __grid_constant__ CUtensorMap tm_y, TcParams p) {
  using K = Cfg<R, NS>;
  constexpr int Q = K::Q, KP = K::KP, TG = K::TG, TPG = K::TPG, HR = K::HR;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_addr(smem);

  __shared__ uint64_t bar_x[2], bar_m1, bar_m3;
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_flag;
  __shared__ float s_lam2[64], s_gam[64], s_wp[64], s_wend[64], s_eL[64], s_dt[64];
  __shared__ float s_tot[2][TG][KP];    // per token group: angle total (hi, lo)
  __shared__ float s_carry[2][2][KP];   // [parity][hi, lo][pair]: angle before the chunk
  __shared__ float s_eLend, s_wmax;
  __shared__ float s_red[3][kWarps];   // per-warp maxima: |B|, |C|, |x|
  __shared__ float s_hred[kWarps];     // per-warp maxima of |H|
  __shared__ float s_bias_red[2][kWarps];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t H = p.H, L = p.L, G = p.G;
  const int64_t bh = blockIdx.x, b = bh / H, h = bh % H, g = h / (H / G);
  const float A_h = p.A[h];
  const int nC = p.nchunks;

  // ---------------------------------------------------------------- setup
  if (warp == 0) {
    ptx::tmem_alloc(&tmem_holder, kTmemCols);
    ptx::tmem_relinquish();
  }
  if (tid == 0) {
    abort_flag = 0;
    ptx::mbar_init(&bar_x[0], 1);
    ptx::mbar_init(&bar_x[1], 1);
    ptx::mbar_init(&bar_m1, 1);
    ptx::mbar_init(&bar_m3, 1);
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&tm_x);
    ptx::prefetch_tensormap(&tm_y);
  }
  for (int i = tid; i < 4 * KP; i += kThreads) (&s_carry[0][0][0])[i] = 0.f;
  // zero fp16 state copy: the entering state of chunk 0
  for (uint32_t i = tid * 16; i < (uint32_t)NS * 128u; i += kThreads * 16)
    sts128(sbase + K::kH + i, make_uint4(0, 0, 0, 0));

  // per-thread constants of the angle phase: pair k, token group tq
  const int kq = tid % KP, tq = tid / KP;
  float bbias[2][R], cbias[2][R];
  float bmax_bias = 0.f, cmax_bias = 0.f;
#pragma unroll
  for (int e = 0; e < 2; ++e)
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int64_t ix = (h * NS + 2 * kq + e) * R + r;
      bbias[e][r] = p.B_bias ? p.B_bias[ix] : 0.f;
      cbias[e][r] = p.C_bias ? p.C_bias[ix] : 0.f;
      bmax_bias = fmaxf(bmax_bias, fabsf(bbias[e][r]));
      cmax_bias = fmaxf(cmax_bias, fabsf(cbias[e][r]));
    }
  bmax_bias = warp_max(bmax_bias);
  cmax_bias = warp_max(cmax_bias);
  if (lane == 0) {
    s_bias_red[0][warp] = bmax_bias;
    s_bias_red[1][warp] = cmax_bias;
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem = tmem_holder;
  bmax_bias = 0.f;
  cmax_bias = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    bmax_bias = fmaxf(bmax_bias, s_bias_red[0][w]);
    cmax_bias = fmaxf(cmax_bias, s_bias_red[1][w]);
  }
  constexpr uint32_t kXBytes = (uint32_t)(Q * kP * R * 2);
  if (tid == 0) {
    for (int c = 0; c < 2 && c < nC; ++c) {
      ptx::mbar_arrive_expect_tx(&bar_x[c], kXBytes);
      ptx::tma_load_4d(smem + K::kXs + c * kTileBytes, &tm_x, &bar_x[c], 0, (int)h, c * Q, (int)b);
    }
  }

  // state ownership (D accumulator layout): quadrant of the warp and column half
  const int quad = warp & 3, chalf = warp >> 2;
  float hreg[HR];
#pragma unroll
  for (int i = 0; i < HR; ++i) hreg[i] = 0.f;
  float h_inv_prev = 1.f;  // 1/sigma of the fp16 state copy the next Yoff reads

  const __nv_bfloat16* Bg = p.B;
  const __nv_bfloat16* Cg = p.C;

  for (int c = 0; c < nC; ++c) {
    const int64_t t0 = (int64_t)c * Q;
    const int stage = c & 1;
    // ---------------------------------------------------- phase 0: decay scan
    if (warp == 0) {
      float dtv[2], lmv[2], bnx[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int i = lane + 32 * j;
        const int64_t t = t0 + i;
        dtv[j] = 0.f; lmv[j] = 0.f; bnx[j] = 0.f;
        if (i < Q && t < L) {
          dtv[j] = p.dt[(b * L + t) * H + h];
          lmv[j] = p.lam[(b * L + t) * H + h];
          if (t + 1 < L)
            bnx[j] = (1.f - p.lam[(b * L + t + 1) * H + h]) * p.dt[(b * L + t + 1) * H + h];
        }
      }
      // inclusive prefix of Delta*A (in log2 units) over the chunk
      float a0 = dtv[0] * A_h * kLog2e, a1 = dtv[1] * A_h * kLog2e;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float v0 = __shfl_up_sync(0xffffffffu, a0, o);
        const float v1 = __shfl_up_sync(0xffffffffu, a1, o);
        if (lane >= o) { a0 += v0; a1 += v1; }
      }
      a1 += __shfl_sync(0xffffffffu, a0, 31);
      const float lam_end = (Q <= 32) ? __shfl_sync(0xffffffffu, a0, Q - 1)
                                      : __shfl_sync(0xffffffffu, a1, (Q - 1) & 31);
      float lv[2] = {a0, a1};
      float wm = 0.f;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int i = lane + 32 * j;
        if (i < Q) {
          const float gam = lmv[j] * dtv[j];
          const float wpv = gam + bnx[j];
          const float we = exp2f(lam_end - lv[j]) * wpv;
          s_lam2[i] = lv[j];
          s_gam[i] = gam;
          s_wp[i] = wpv;
          s_wend[i] = we;
          s_eL[i] = exp2f(lv[j]);
          s_dt[i] = dtv[j];
          wm = fmaxf(wm, fabsf(we));
        }
      }
      wm = warp_max(wm);
      if (lane == 0) {
        s_eLend = exp2f(lam_end);
        s_wmax = wm;
      }
    }
    // raw loads of this thread's tokens (B, C pairs for all ranks; theta)
    float th[TPG];
    uint32_t braw[TPG][R], craw[TPG][R];
    float bmax = 0.f, cmax = 0.f;
#pragma unroll
    for (int i = 0; i < TPG; ++i) {
      const int64_t t = t0 + tq * TPG + i;
      th[i] = 0.f;
#pragma unroll
      for (int r = 0; r < R; ++r) { braw[i][r] = 0u; craw[i][r] = 0u; }
      if (t < L) {
        th[i] = p.theta[((b * L + t) * G + g) * KP + kq];
        const int64_t base = ((b * L + t) * G + g) * (int64_t)NS * R + (int64_t)(2 * kq) * R;
        if constexpr (R == 1) {
          braw[i][0] = *reinterpret_cast<const uint32_t*>(Bg + base);
          craw[i][0] = *reinterpret_cast<const uint32_t*>(Cg + base);
        } else if constexpr (R == 2) {
          const uint2 vb = *reinterpret_cast<const uint2*>(Bg + base);
          const uint2 vc = *reinterpret_cast<const uint2*>(Cg + base);
          braw[i][0] = vb.x; braw[i][1] = vb.y;
          craw[i][0] = vc.x; craw[i][1] = vc.y;
        } else {
          const uint4 vb = *reinterpret_cast<const uint4*>(Bg + base);
          const uint4 vc = *reinterpret_cast<const uint4*>(Cg + base);
          braw[i][0] = vb.x; braw[i][1] = vb.y; braw[i][2] = vb.z; braw[i][3] = vb.w;
          craw[i][0] = vc.x; craw[i][1] = vc.y; craw[i][2] = vc.z; craw[i][3] = vc.w;
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        bmax = fmaxf(bmax, bf_absmax(braw[i][r]));
        cmax = fmaxf(cmax, bf_absmax(craw[i][r]));
      }
    }
    __syncthreads();  // decay scan visible
    // ---------------------------------------------------- phase 1: angles, RoPE fold
    // cumulative angle over this thread's tokens (radians), with Kahan's
    // compensation so that the chunk-to-chunk carry does not drift over long
    // sequences; ph[i] is the plain running sum, total = run - comp
    float ph[TPG];
    float run = 0.f, comp = 0.f;
#pragma unroll
    for (int i = 0; i < TPG; ++i) {
      const float yk = __fmul_rn(s_dt[tq * TPG + i], th[i]) - comp;
      const float tk = run + yk;
      comp = (tk - run) - yk;
      run = tk;
      ph[i] = run;
    }
    s_tot[0][tq][kq] = run;
    s_tot[1][tq][kq] = -comp;
    // this chunk's x tile: wait for its TMA, read this thread's part, bound |x|
    const bool x_ok = wait_or_abort(&bar_x[stage], (uint32_t)((c >> 1) & 1), &abort_flag, p.status);
    const uint32_t xs = sbase + K::kXs + stage * kTileBytes;
    constexpr int kXItems = (R == 1) ? 2 : (Q * (kP / 4)) / kThreads;  // per thread
    uint4 xv[kXItems][(R == 1) ? 1 : R / 2];
    float xmax = 0.f;
    if (x_ok) {
#pragma unroll
      for (int j = 0; j < kXItems; ++j) {
        const int it = tid + kThreads * j;
        if constexpr (R == 1) {
          xv[j][0] = lds128(xs + (uint32_t)it * 16u);  // 16-byte chunk `it`, row it / 8
        } else {
          // raw x tile [token][p][r]; item = (token s, block of 4 p): 8R bytes
          const int s = it / (kP / 4), pb = it % (kP / 4);
          const uint32_t src = xs + (uint32_t)(s * kP * R + 4 * pb * R) * 2u;
#pragma unroll
          for (int q2 = 0; q2 < R / 2; ++q2) xv[j][q2] = lds128(src + 16u * q2);
        }
#pragma unroll
        for (int q2 = 0; q2 < ((R == 1) ? 1 : R / 2); ++q2) {
          xmax = fmaxf(xmax, fmaxf(fmaxf(bf_absmax(xv[j][q2].x), bf_absmax(xv[j][q2].y)),
                                   fmaxf(bf_absmax(xv[j][q2].z), bf_absmax(xv[j][q2].w))));
        }
      }
    }
    bmax = warp_max(bmax);
    cmax = warp_max(cmax);
    xmax = warp_max(xmax);
    if (lane == 0) {
      s_red[0][warp] = bmax;
      s_red[1][warp] = cmax;
      s_red[2][warp] = xmax;
    }
    __syncthreads();
    if (abort_flag) break;
    // per-chunk fp16 scales of the rotated B / C tiles and of w X
    float sigB, invB, sigC, invC, sigX, invX;
    {
      float mb = 0.f, mc = 0.f, mx = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        mb = fmaxf(mb, s_red[0][w]);
        mc = fmaxf(mc, s_red[1][w]);
        mx = fmaxf(mx, s_red[2][w]);
      }
      // a rotated pair keeps its norm: |Rot(v)_i| <= sqrt(2) max|v| < 2 max|v|
      pow2_scale(2.f * (mb + bmax_bias), &sigB, &invB);
      pow2_scale(2.f * (mc + cmax_bias), &sigC, &invC);
      pow2_scale(mx * s_wmax, &sigX, &invX);
    }
    // angle before this thread's first token: carry + earlier groups (float-float)
    float oh = s_carry[stage][0][kq], ol = s_carry[stage][1][kq];
    for (int q2 = 0; q2 < tq; ++q2) ff_add(oh, ol, s_tot[0][q2][kq], s_tot[1][q2][kq]);
    ff_wrap(oh, ol);
    if (tq == TG - 1) {
      float eh = oh, el = ol;
      ff_add(eh, el, run, -comp);
      ff_wrap(eh, el);
      s_carry[stage ^ 1][0][kq] = eh;
      s_carry[stage ^ 1][1][kq] = el;
    }
#pragma unroll
    for (int i = 0; i < TPG; ++i) {
      float ang = oh + (ol + ph[i]);
      const float kw = rintf(ang * kInvTwoPi);
      ang = fmaf(-kw, kPi2a, ang);
      ang = fmaf(-kw, kPi2b, ang);
      float sn, cs;
      __sincosf(ang, &sn, &cs);
      const float csB = cs * sigB, snB = sn * sigB, csC = cs * sigC, snC = sn * sigC;
      const int t = tq * TPG + i;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        // word layout of the 2R raw values: n = 2k at r, then n = 2k + 1 at r
        float b0, b1, c0, c1;
        if constexpr (R == 1) {
          b0 = bf_lo(braw[i][0]); b1 = bf_hi(braw[i][0]);
          c0 = bf_lo(craw[i][0]); c1 = bf_hi(craw[i][0]);
        } else {
          const int w0 = r >> 1, w1 = (R >> 1) + (r >> 1);
          b0 = (r & 1) ? bf_hi(braw[i][w0]) : bf_lo(braw[i][w0]);
          b1 = (r & 1) ? bf_hi(braw[i][w1]) : bf_lo(braw[i][w1]);
          c0 = (r & 1) ? bf_hi(craw[i][w0]) : bf_lo(craw[i][w0]);
          c1 = (r & 1) ? bf_hi(craw[i][w1]) : bf_lo(craw[i][w1]);
        }
        b0 += bbias[0][r]; b1 += bbias[1][r];
        c0 += cbias[0][r]; c1 += cbias[1][r];
        // sigma Rot(-Phi) = sigma [[cos, sin], [-sin, cos]]
        const float bt0 = fmaf(csB, b0, snB * b1), bt1 = fmaf(csB, b1, -snB * b0);
        const float ct0 = fmaf(csC, c0, snC * c1), ct1 = fmaf(csC, c1, -snC * c0);
        const uint32_t row = (uint32_t)(t * R + r);
        const uint32_t o = tile_off(row, 2u * kq, 64u);
        sts32(sbase + K::kBt + o, pack_f16(bt0, bt1));
        sts32(sbase + K::kCt + o, pack_f16(ct0, ct1));
      }
    }
    // w X (fp16, scaled) and, for R > 1, X re-laid as [(token, rank)][p] (bf16)
#pragma unroll
    for (int j = 0; j < kXItems; ++j) {
      const int it = tid + kThreads * j;
      if constexpr (R == 1) {
        const uint32_t row = (uint32_t)it >> 3;
        const float w = s_wend[row] * sigX;
        const uint4 v = xv[j][0];
        sts128(sbase + K::kXw + (uint32_t)it * 16u,
               make_uint4(pack_f16(w * bf_lo(v.x), w * bf_hi(v.x)),
                          pack_f16(w * bf_lo(v.y), w * bf_hi(v.y)),
                          pack_f16(w * bf_lo(v.z), w * bf_hi(v.z)),
                          pack_f16(w * bf_lo(v.w), w * bf_hi(v.w))));
      } else {
        const int s = it / (kP / 4), pb = it % (kP / 4);
        uint32_t wv[2 * R];
#pragma unroll
        for (int q2 = 0; q2 < R / 2; ++q2) {
          wv[4 * q2] = xv[j][q2].x; wv[4 * q2 + 1] = xv[j][q2].y;
          wv[4 * q2 + 2] = xv[j][q2].z; wv[4 * q2 + 3] = xv[j][q2].w;
        }
        const float w = s_wend[s] * sigX;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          float v4[4];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int e = q4 * R + r;  // element index within the 4R values
            v4[q4] = (e & 1) ? bf_hi(wv[e >> 1]) : bf_lo(wv[e >> 1]);
          }
          const uint32_t row = (uint32_t)(s * R + r);
          const uint32_t o = sw128(row, 4u * pb);
          sts64(sbase + K::kXb + o, pack_bf16(v4[0], v4[1]), pack_bf16(v4[2], v4[3]));
          sts64(sbase + K::kXw + o, pack_f16(w * v4[0], w * v4[1]), pack_f16(w * v4[2], w * v4[3]));
        }
      }
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    // ---------------------------------------------------- phase 2: S, D, Yoff
    const uint32_t xop = (R == 1) ? xs : (sbase + K::kXb);
    if (tid == 0) {
      constexpr uint32_t idS = ptx::idesc_f16_f32(64, 64, false, false);
      constexpr uint32_t idD = ptx::idesc_f16_f32(NS, 64, true, true);
      constexpr uint32_t idYo = ptx::idesc_f16_f32(64, 64, false, true);
#pragma unroll
      for (int kk = 0; kk < NS / 16; ++kk)
        ptx::mma_bf16_ss(tmem + kColS, desc_k(sbase + K::kCt, kk, 64), desc_k(sbase + K::kBt, kk, 64),
                         idS, kk > 0);
#pragma unroll
      for (int kk = 0; kk < kQR / 16; ++kk)
        ptx::mma_bf16_ss(tmem + kColD, desc_mn(sbase + K::kBt, kk, 64u * 128u),
                         desc_mn(sbase + K::kXw, kk, 64u * 128u), idD, kk > 0);
#pragma unroll
      for (int kk = 0; kk < NS / 16; ++kk)
        ptx::mma_bf16_ss(tmem + kColYo, desc_k(sbase + K::kCt, kk, 64),
                         desc_mn(sbase + K::kH, kk, (uint32_t)NS * 128u), idYo, kk > 0);
      ptx::mma_commit(&bar_m1);
    }
    __syncwarp();
    // ---------------------------------------------------- phase 3: mask, state
    const bool m1_ok = wait_or_abort(&bar_m1, (uint32_t)(c & 1), &abort_flag, p.status);
    ptx::tc_fence_after_sync();
    float hmax = 0.f;
    if (m1_ok) {
      // masked scores: thread -> row a, 16 consecutive columns (M=64 layout)
      {
        uint32_t sv[16];
        ptx::tmem_ld16_16x32bx2<16>(tmem + kColS + ((uint32_t)(32 * quad) << 16) + 32u * chalf, sv);
        ptx::tmem_ld_wait(sv);
        const int a = 16 * quad + (lane & 15);
        const int c0 = 32 * chalf + 16 * (lane >> 4);
        const int t = a / R;
        const float invBC = invB * invC;
        const float lt = s_lam2[t];
        uint32_t ph_[8], pl_[8];
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          float hi2[2], lo2[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int s = (c0 + j + e) / R;
            float m = 0.f;
            if (s < t) m = exp2f(lt - s_lam2[s]) * s_wp[s];
            else if (s == t) m = s_gam[s];
            const float v = (m * invBC) * __uint_as_float(sv[j + e]);
            const float vh = __bfloat162float(__float2bfloat16_rn(v));
            hi2[e] = vh;
            lo2[e] = v - vh;
          }
          ph_[j >> 1] = pack_bf16(hi2[0], hi2[1]);
          pl_[j >> 1] = pack_bf16(lo2[0], lo2[1]);
        }
        const uint32_t o0 = sw128((uint32_t)a, (uint32_t)c0);
        const uint32_t o1 = sw128((uint32_t)a, (uint32_t)c0 + 8u);
        sts128(sbase + K::kPh + o0, make_uint4(ph_[0], ph_[1], ph_[2], ph_[3]));
        sts128(sbase + K::kPh + o1, make_uint4(ph_[4], ph_[5], ph_[6], ph_[7]));
        sts128(sbase + K::kPl + o0, make_uint4(pl_[0], pl_[1], pl_[2], pl_[3]));
        sts128(sbase + K::kPl + o1, make_uint4(pl_[4], pl_[5], pl_[6], pl_[7]));
      }
      // state: H = exp(Lam_end) H + D / (sigma_B sigma_X)
      {
        const float eend = s_eLend;
        const float invBX = invB * invX;
        if constexpr (NS == 128) {
          // M=128 layout: lane = row n; this warp owns p in [32*chalf, +32)
          uint32_t d0[16], d1[16];
          const uint32_t ta = tmem + kColD + ((uint32_t)(32 * quad) << 16) + 32u * chalf;
          ptx::tmem_ld16(ta, d0);
          ptx::tmem_ld16(ta + 16, d1);
          ptx::tmem_ld_wait(d0);
          ptx::tmem_ld_wait(d1);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            hreg[j] = fmaf(invBX, __uint_as_float(d0[j]), eend * hreg[j]);
            hreg[16 + j] = fmaf(invBX, __uint_as_float(d1[j]), eend * hreg[16 + j]);
          }
        } else {
          // M=64 layout: row n = 16*quad + (lane & 15); 16 columns per thread
          uint32_t d0[16];
          ptx::tmem_ld16_16x32bx2<16>(tmem + kColD + ((uint32_t)(32 * quad) << 16) + 32u * chalf, d0);
          ptx::tmem_ld_wait(d0);
#pragma unroll
          for (int j = 0; j < 16; ++j) hreg[j] = fmaf(invBX, __uint_as_float(d0[j]), eend * hreg[j]);
        }
#pragma unroll
        for (int j = 0; j < HR; ++j) hmax = fmaxf(hmax, fabsf(hreg[j]));
      }
    }
    hmax = warp_max(hmax);
    if (lane == 0) s_hred[warp] = hmax;
    if (tid == 0) ptx::tma_store_wait_read<0>();  // output staging free again
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (abort_flag) break;
    ptx::tc_fence_after_sync();
    // ---------------------------------------------------- phase 4: Y = P X
    if (tid == 0) {
      constexpr uint32_t idY = ptx::idesc_bf16_f32(64, 64, false, true);
#pragma unroll
      for (int kk = 0; kk < kQR / 16; ++kk)
        ptx::mma_bf16_ss(tmem + kColY, desc_k(sbase + K::kPh, kk, 64), desc_mn(xop, kk, 64u * 128u),
                         idY, kk > 0);
#pragma unroll
      for (int kk = 0; kk < kQR / 16; ++kk)
        ptx::mma_bf16_ss(tmem + kColY, desc_k(sbase + K::kPl, kk, 64), desc_mn(xop, kk, 64u * 128u),
                         idY, 1u);
      ptx::mma_commit(&bar_m3);
    }
    __syncwarp();
    // fp16 copy of the new state for the next chunk's Ct H_in product (its
    // previous copy was last read by this chunk's Yoff MMA, complete above)
    float h_sig, h_inv;
    {
      float m = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) m = fmaxf(m, s_hred[w]);
      pow2_scale(m, &h_sig, &h_inv);
      if constexpr (NS == 128) {
        const uint32_t n = (uint32_t)(32 * quad + lane);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const float* hv = hreg + 8 * q4;
          sts128(sbase + K::kH + sw128(n, 32u * chalf + 8u * q4),
                 make_uint4(pack_f16(h_sig * hv[0], h_sig * hv[1]), pack_f16(h_sig * hv[2], h_sig * hv[3]),
                            pack_f16(h_sig * hv[4], h_sig * hv[5]), pack_f16(h_sig * hv[6], h_sig * hv[7])));
        }
      } else {
        const uint32_t n = (uint32_t)(16 * quad + (lane & 15));
        const uint32_t cb = 32u * chalf + 16u * (lane >> 4);
#pragma unroll
        for (int q4 = 0; q4 < 2; ++q4) {
          const float* hv = hreg + 8 * q4;
          sts128(sbase + K::kH + sw128(n, cb + 8u * q4),
                 make_uint4(pack_f16(h_sig * hv[0], h_sig * hv[1]), pack_f16(h_sig * hv[2], h_sig * hv[3]),
                            pack_f16(h_sig * hv[4], h_sig * hv[5]), pack_f16(h_sig * hv[6], h_sig * hv[7])));
        }
      }
    }
    const bool m3_ok = wait_or_abort(&bar_m3, (uint32_t)(c & 1), &abort_flag, p.status);
    ptx::tc_fence_after_sync();
    // x stage of this chunk is free: prefetch chunk c + 2 into it
    if (tid == 0 && m3_ok && c + 2 < nC) {
      ptx::mbar_arrive_expect_tx(&bar_x[stage], kXBytes);
      ptx::tma_load_4d(smem + K::kXs + stage * kTileBytes, &tm_x, &bar_x[stage], 0, (int)h,
                       (c + 2) * Q, (int)b);
    }
    // ---------------------------------------------------- phase 5: outputs
    if (m3_ok) {
      uint32_t yv[16], yo[16];
      const uint32_t ta = ((uint32_t)(32 * quad) << 16) + 32u * chalf;
      ptx::tmem_ld16_16x32bx2<16>(tmem + kColY + ta, yv);
      ptx::tmem_ld16_16x32bx2<16>(tmem + kColYo + ta, yo);
      ptx::tmem_ld_wait(yv);
      ptx::tmem_ld_wait(yo);
      const int a = 16 * quad + (lane & 15);
      const int c0 = 32 * chalf + 16 * (lane >> 4);  // first p of this thread
      const float el = s_eL[a / R] * (invC * h_inv_prev);
      float y[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) y[j] = fmaf(el, __uint_as_float(yo[j]), __uint_as_float(yv[j]));
      if constexpr (R == 1) {
        const uint32_t o0 = sw128((uint32_t)a, (uint32_t)c0);
        const uint32_t o1 = sw128((uint32_t)a, (uint32_t)c0 + 8u);
        sts128(sbase + K::kYs + o0, make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]),
                                               pack_bf16(y[4], y[5]), pack_bf16(y[6], y[7])));
        sts128(sbase + K::kYs + o1, make_uint4(pack_bf16(y[8], y[9]), pack_bf16(y[10], y[11]),
                                               pack_bf16(y[12], y[13]), pack_bf16(y[14], y[15])));
      } else {
        // staging in the global layout of one chunk: [token][p][r]
        const int t = a / R, r = a % R;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          __nv_bfloat16 v = __float2bfloat16_rn(y[j]);
          sts16(sbase + K::kYs + (uint32_t)((t * kP + c0 + j) * R + r) * 2u,
                *reinterpret_cast<uint16_t*>(&v));
        }
      }
    }
    h_inv_prev = h_inv;
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (abort_flag) break;
    if (tid == 0) {
      ptx::tma_store_4d(&tm_y, smem + K::kYs, 0, (int)h, (int)t0, (int)b);
      ptx::tma_store_commit();
    }
  }

  // ---------------------------------------------------------------- final state
  if (tid == 0) ptx::tma_store_wait_all<0>();
  if (!abort_flag && p.final_state) {
    // explicit frame: h = Rot(Phi_{L-1}) g, rows (2k, 2k+1)
    float* fs = p.final_state + bh * (int64_t)NS * kP;
    const float* carry_h = s_carry[nC & 1][0];
    const float* carry_l = s_carry[nC & 1][1];
    if constexpr (NS == 128) {
      const int n = 32 * quad + lane;
      float sn, cs;
      sincosf(carry_h[n >> 1] + carry_l[n >> 1], &sn, &cs);
      const bool odd = n & 1;
      float outv[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float other = __shfl_xor_sync(0xffffffffu, hreg[j], 1);
        // even row: c*g0 - s*g1 ; odd row: s*g0 + c*g1
        outv[j] = odd ? fmaf(sn, other, cs * hreg[j]) : fmaf(-sn, other, cs * hreg[j]);
      }
      float4* dst = reinterpret_cast<float4*>(fs + (int64_t)n * kP + 32 * chalf);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        dst[j] = make_float4(outv[4 * j], outv[4 * j + 1], outv[4 * j + 2], outv[4 * j + 3]);
    } else {
      const int n = 16 * quad + (lane & 15);
      float sn, cs;
      sincosf(carry_h[n >> 1] + carry_l[n >> 1], &sn, &cs);
      const bool odd = n & 1;
      float outv[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float other = __shfl_xor_sync(0xffffffffu, hreg[j], 1);
        outv[j] = odd ? fmaf(sn, other, cs * hreg[j]) : fmaf(-sn, other, cs * hreg[j]);
      }
      float4* dst = reinterpret_cast<float4*>(fs + (int64_t)n * kP + 32 * chalf + 16 * (lane >> 4));
#pragma unroll
      for (int j = 0; j < 4; ++j)
        dst[j] = make_float4(outv[4 * j], outv[4 * j + 1], outv[4 * j + 2], outv[4 * j + 3]);
    }
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// x / out as a 4-D tensor {P*R, H, L, b}; the box is one head's chunk.
bool make_act_map(CUtensorMap* m, const void* ptr, const ScanArgs& a) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const uint64_t PR = (uint64_t)a.P * a.R;
  cuuint64_t dims[4] = {PR, (cuuint64_t)a.H, (cuuint64_t)a.L, (cuuint64_t)a.batch};
  cuuint64_t strides[3] = {PR * 2, PR * 2 * a.H, PR * 2 * a.H * a.L};
  const uint32_t Q = (uint32_t)a.Q;
  cuuint32_t box[4] = {(cuuint32_t)PR, 1, Q, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapSwizzle sw = (a.R == 1) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int R, int NS>
cudaError_t launch_rn(const ScanArgs& a, unsigned int* status, cudaStream_t s) {
  CUtensorMap tx, ty;
  if (!make_act_map(&tx, a.x, a) || !make_act_map(&ty, a.out, a)) return cudaErrorInvalidValue;
  TcParams p;
  p.dt = a.dt; p.A = a.A; p.lam = a.lam;
  p.B = static_cast<const __nv_bfloat16*>(a.B);
  p.C = static_cast<const __nv_bfloat16*>(a.C);
  p.theta = a.theta; p.B_bias = a.B_bias; p.C_bias = a.C_bias;
  p.final_state = a.final_state; p.status = status;
  p.L = a.L; p.H = a.H; p.G = a.G;
  p.nchunks = (int)((a.L + a.Q - 1) / a.Q);
  constexpr uint32_t smem = Cfg<R, NS>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(scan_tc_kernel<R, NS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  scan_tc_kernel<R, NS><<<(unsigned)(a.batch * a.H), kThreads, smem, s>>>(tx, ty, p);
  return cudaGetLastError();
}

}  // namespace

bool scan_tc_supported(int64_t N, int64_t P, int R, int Q) {
  if (P != kP) return false;
  if (N != 64 && N != 128) return false;
  if (!(R == 1 || R == 2 || R == 4)) return false;
  return Q * R == kQR;
}

cudaError_t launch_scan_tc(const ScanArgs& a, unsigned int* status, cudaStream_t s) {
  if (a.L > 0x7fffffffLL - 2 * kQR || a.batch > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int key = a.R * 1000 + (int)a.N;
  switch (key) {
    case 1064: return launch_rn<1, 64>(a, status, s);
    case 1128: return launch_rn<1, 128>(a, status, s);
    case 2064: return launch_rn<2, 64>(a, status, s);
    case 2128: return launch_rn<2, 128>(a, status, s);
    case 4064: return launch_rn<4, 64>(a, status, s);
    case 4128: return launch_rn<4, 128>(a, status, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace m3
