// Tensor-core (tcgen05 + TMEM + TMA) chunked prefill of the Mamba-3 scan.
//
// Scope: bf16 activations, head dim P = 64, state N in {64, 128}, MIMO rank
// R in {1, 2, 4} with chunk Q = 64 / R, so that the flattened (token, rank)
// tile of a chunk has QR = 64 rows (the MIMO chunk rule C_MIMO = C_SISO / R of
// "Mamba-3: Improved Sequence Modeling using State Space Principles",
// papernotes.org, sec. 3 MIMO).
//
// Math (per batch row b and head h). The rotation of the complex-valued state
// is folded into B and C as a cumulative data-dependent RoPE ("MAMBA-3:
// IMPROVED SEQUENCE MODELING USING STATE SPACE PRINCIPLES", aipaper.cc,
// sec. 4.2, Prop. 3): with Phi_t = sum_{u<=t} Delta_u theta_u (per state pair,
// over the whole sequence) and Rot(-Phi_t) applied to B_t and C_t,
//   g_t = alpha_t g_{t-1} + beta_t Bt_{t-1} x_{t-1}^T + gamma_t Bt_t x_t^T,
//   y_t = Ct_t^T g_t,   h_t = Rot(Phi_t) g_t   (explicit frame).
// The exponential-trapezoidal weights are those of Prop. 1 (same page,
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
// end).
//
// Precision. The rotated operands are data derived in fp32, not inputs, and
// the score matrix sums products much larger than y itself (|B|^2 = N for
// RMS-normalised B). Their operand tiles (Bt, Ct, w X and the state copy) are
// therefore fp16 (11-bit significand, kind::f16 MMA with fp32 accumulation),
// each scaled by a power of two chosen per chunk from a bound of its
// magnitude, so fp16's range never limits the inputs. The scales are undone
// exactly where a per-element factor is applied anyway (mask, state rescale,
// output). P and the X operand of P X are fp16 too (X scaled by a power of
// two: exact for bf16 inputs), so that P keeps the same 11 bits as the
// operands it is made from. The cumulative angle is carried
// from chunk to chunk as a float-float pair, so it does not drift over long
// sequences.
//
// Organisation: a persistent CTA of 256 threads (8 warps) walks work units
// (whole (b, h) sequences, or segments of them when there are fewer sequences
// than SMs) chunk by chunk; two CTAs share an SM (about 104 KB of shared
// memory and 256 TMEM columns each), so one CTA's barriers and MMA waits are
// covered by the other's work. Every warp takes part in every phase of a chunk:
//   fold   raw B, C, x tiles (TMA, refilled with the next chunk as soon as they
//          are read) -> magnitude bounds and per-token-group angle sums ->
//          barrier -> fp16 scales, angle offsets, sincos, RoPE fold of B and C
//          into 128-byte-swizzled fp16 UMMA tiles, w X, the fp16 X operand, and
//          the rescale of the state held in TMEM by exp(Lam_end) and the change
//          of scale -> barrier -> one thread (lane 0 of warp 5) issues D
//          (accumulated onto the state), S and Yoff = Ct H_in; every thread
//          then issues its loads of the next chunk's theta (and warp 4 those
//          of the decay inputs)
//   mask   S -> P (fp16, scaled; over the Bt tile, which D and S no longer
//          read) -> barrier -> one thread issues Y = P X
//   state  the state after D (TMEM) -> its bound -> barrier -> its scaled fp16
//          copy for the next chunk's Yoff
//   output y = Y + exp(Lam_t) Yoff -> bf16 -> global memory (16-byte stores;
//          a TMA store from a staging tile for R > 1); final state
// The fp32 state lives in the TMEM columns of the D accumulator: each chunk
// rescales it in place and the D MMA accumulates onto it. One warp computes
// the next chunk's decay scan (warp shuffles), in the mask phase; theta is
// read from global memory into registers one chunk ahead.
// Every mbarrier wait is bounded; on expiry the CTA records the status word,
// every thread leaves the loop at the next block barrier, and the CTA still
// waits for its copies in flight and frees its tensor memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace m3 {
namespace {

constexpr int kThreads = 256;  // 8 warps, two CTAs per SM (128 registers per thread)
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
// sin.approx / cos.approx keep their accuracy for arguments up to 100 pi;
// angles beyond this bound are reduced first.
constexpr float kAngleDirect = 300.f;

// TMEM column offsets of the four fp32 accumulators. D holds the state.
constexpr uint32_t kColS = 0, kColD = 64, kColY = 128, kColYo = 192;

constexpr uint32_t align1k(uint32_t v) { return (v + 1023u) & ~1023u; }

// F32: the fp32 precision mode. Activations arrive as fp32; every operand
// tile is a pair of fp16 tiles, high part and residual (v = hi + lo to ~22
// bits), and each product is formed from three MMAs (hi hi + hi lo + lo hi).
template <int R, int NS, bool F32 = false>
struct Cfg {
  static constexpr int Q = kQR / R;          // tokens per chunk
  static constexpr int KP = NS / 2;          // rotating state pairs
  static constexpr int KP2 = KP / 2;         // pair-pairs: a fold thread owns two pairs
  static constexpr int TG = kThreads / KP2;  // token groups of the fold
  static constexpr int TPG = Q / TG;         // tokens per fold thread
  static_assert(TPG >= 1 && Q % TG == 0, "token groups must divide the chunk");
  static constexpr int HR = NS * kP / kThreads;  // fp32 state values per thread
  static constexpr int AB = F32 ? 4 : 2;           // bytes per raw activation element
  static constexpr int BW = 4 * R * AB / 4;  // raw 32-bit words of B (or C) per token and thread
  static constexpr int XW = (R == 1 ? 8 : 4 * R) * AB / 4;  // raw x words per item
  static constexpr int OPS = F32 ? 2 : 1;  // fp16 tiles per operand (hi, lo)
  // raw slot (TMA destination): B, C [Q][NS*R], x [Q][P*R] (bf16: x 128B-swizzled for R = 1)
  static constexpr uint32_t kRawB = 0;
  static constexpr uint32_t kRawC = kRawB + Q * NS * R * AB;
  static constexpr uint32_t kRawX = align1k(kRawC + Q * NS * R * AB);
  static constexpr uint32_t kRawEnd = kRawX + (uint32_t)(Q * kP * R * AB);
  // operand tiles: Bt, Ct [64][NS] fp16, w X [64][64] fp16, X [64][64] fp16,
  // the fp16 state copy [NS][64]; F32: each followed by its residual
  static constexpr uint32_t kBtLo = 64 * NS * 2;   // hi -> lo offset of Bt, Ct
  static constexpr uint32_t kXLo = kTileBytes;     // ... of w X, X, P
  static constexpr uint32_t kHLo = NS * 128;       // ... of the state copy
  static_assert(kBtLo % 1024 == 0 && kXLo % 1024 == 0 && kHLo % 1024 == 0,
                "residual tiles keep the 1024-byte alignment of the swizzle atom");
  static constexpr uint32_t kBt = align1k(kRawEnd);
  static constexpr uint32_t kCt = kBt + OPS * 64 * NS * 2;
  static constexpr uint32_t kXw = kCt + OPS * 64 * NS * 2;
  static constexpr uint32_t kXo = kXw + OPS * kTileBytes;
  static constexpr uint32_t kH = kXo + OPS * kTileBytes;
  static constexpr uint32_t kHEnd = kH + OPS * NS * 128;
  // masked scores P (F32: high and low parts): over Bt when it is large enough
  static constexpr uint32_t kPh = (NS == 128 || F32) ? kBt : kHEnd;
  static constexpr uint32_t kPl = kPh + kTileBytes;
  static constexpr uint32_t kPEnd = F32 ? kPl + kTileBytes : kPl;
  // output staging (R > 1): over w X (hi, lo), which only D reads
  static constexpr uint32_t kYs = kXw;
  static constexpr uint32_t kBytes = (kPEnd > kHEnd) ? kPEnd : kHEnd;
  static constexpr uint32_t kSmem = kBytes + 1024;  // + alignment slack
  // bytes landing on the raw barrier per chunk (full pass; state-only pass)
  static constexpr uint32_t kTxBytes = 2u * Q * NS * R * AB + (uint32_t)(Q * kP * R * AB);
  static constexpr uint32_t kTxBytesSO = (uint32_t)Q * NS * R * AB + (uint32_t)(Q * kP * R * AB);
};

// Per-chunk scalars (one set per chunk parity): the decay scan's results for
// the chunk's tokens and the chunk's fp16 scales.
struct __align__(16) Scal {
  float lam2[64];  // Lam_t in log2 units
  float gam[64];   // gamma_t
  float wp[64];    // gamma_t + bhat_{t+1}
  float eL[64];    // exp(Lam_t)
  float wend[64];  // exp(Lam_end - Lam_t) (gamma_t + bhat_{t+1})
  float dt[64];    // Delta_t
  float eLend, lamend2, wmax;  // exp(Lam_end), Lam_end (log2), max |wend|
  float invB, invC, invX;      // inverse fp16 scales of Bt, Ct, w X
  float pmul;                  // S -> P units: invB invC times P's scale
  float ykY;                   // Y units -> y: the inverse scales of P and X
  float wpmax;                 // max over the chunk of |gamma_t|, |gamma_t + bhat_{t+1}|
};

struct TcParams {
  const float* dt;
  const float* A;
  const float* lam;
  const float* theta;
  const float* B_bias;
  const float* C_bias;
  void* out;  // bf16, or fp32 in the fp32 mode
  float* final_state;
  unsigned int* status;
  int64_t L, H, G, batch;
  int nchunks;
  // work units are (sequence, segment) pairs of seg_chunks chunks each;
  // nunits = batch * heads * nseg < 2^31, hpg = heads per group
  int seg_chunks, nseg, nunits, heads, hpg;
  // segment passes: the state-only pass writes each unit's local end state to
  // ws_state [unit][N][P] and (log2 decay, angle per pair) to ws_scal
  // [unit][1 + N/2]; the full pass starts unit u from ws_hin[u] (explicit
  // frame) when ws_hin is not NULL
  float* ws_state;
  float* ws_scal;
  const float* ws_hin;
};

__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t col) {
  return row * 128u + ((((col >> 3) ^ row) & 7u) << 4) + (col & 7u) * 2u;
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
// element e of a run of bf16 values packed two per word (little-endian)
template <int N>
__device__ __forceinline__ float bf_at(const uint32_t (&w)[N], int e) {
  return (e & 1) ? bf_hi(w[e >> 1]) : bf_lo(w[e >> 1]);
}
// element e of a token's raw activation words: bf16 pairs, or fp32 (F32)
template <bool F32, int N>
__device__ __forceinline__ float act_at(const uint32_t (&w)[N], int e) {
  if constexpr (F32)
    return __uint_as_float(w[e]);
  else
    return bf_at(w, e);
}
// the fp16 residual pair (a, b) - hi, hi the fp16 pair already formed from (a, b)
__device__ __forceinline__ uint32_t f16_residual(uint32_t hi, float a, float b) {
  const float2 h = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  return pack_f16(a - h.x, b - h.y);
}
// largest magnitude held in an accumulator of bf16x2 abs-maxima, as a float
__device__ __forceinline__ float bf_absmax(uint32_t w) {
  const uint32_t a = w & 0x7fff7fffu;
  return fmaxf(__uint_as_float(a << 16), __uint_as_float(a & 0xffff0000u));
}

// Power of two sigma with M * sigma < 2^15 (inside fp16's range), and 1/sigma;
// sigma is at most 2^(14 - EMIN).
template <int EMIN = -100>
__device__ __forceinline__ void pow2_scale(float M, float* sigma, float* inv) {
  int e = (int)((__float_as_uint(M) >> 23) & 0xffu) - 127;  // M in [2^e, 2^(e+1))
  e = e < EMIN ? EMIN : (e > 127 ? 127 : e);
  *sigma = __uint_as_float((uint32_t)(127 + 14 - e) << 23);
  *inv = __uint_as_float((uint32_t)(127 - 14 + e) << 23);
}

using ptx::add2;
using ptx::fma2;
using ptx::mul2;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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
// Reduce an fp32 angle to about [-pi, pi].
__device__ __forceinline__ float wrap_rad(float a) {
  const float k = rintf(a * kInvTwoPi);
  a = fmaf(-k, kPi2a, a);
  return fmaf(-k, kPi2b, a);
}

// Maximum over the warp of a NON-NEGATIVE float (every use here is a
// magnitude): such floats order like their bit patterns, so one integer
// warp reduction does it.
__device__ __forceinline__ float warp_max(float v) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(v)));
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
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
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
  return v;
}

// A descriptor split into its words; the MMAs of one operand tile differ only
// in the start-address field (low word), so each is the base plus a constant.
struct Desc {
  uint32_t lo, hi;
};
__device__ __forceinline__ Desc make_desc(uint32_t addr, uint32_t lbo) {
  const uint64_t d = ptx::smem_desc_sw128(addr, lbo, 1024u);
  return Desc{(uint32_t)d, (uint32_t)(d >> 32)};
}
// start address advanced by `byte_off` (a multiple of 16, staying in the window)
__device__ __forceinline__ uint64_t desc_at(const Desc& d, uint32_t byte_off) {
  return ((uint64_t)d.hi << 32) | (uint64_t)(d.lo + (byte_off >> 4));
}
// byte offsets of the 16-element K step kk: K-major [rows][K] tiles, MN-major tiles
__host__ __device__ constexpr uint32_t koff_k(int kk, uint32_t rows) {
  return (uint32_t)(kk >> 2) * rows * 128u + (uint32_t)(kk & 3) * 32u;
}
__host__ __device__ constexpr uint32_t koff_mn(int kk) { return (uint32_t)kk * 2048u; }

// Bounded wait on an mbarrier phase; on expiry record the status word and the
// CTA's abort flag. Returns false if the CTA is (now) aborting. Every thread
// that needs the phase waits itself; threads leave the chunk loop only right
// after a block barrier, where the flag reads the same for all of them.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, int* abort_flag,
                                              unsigned int* status) {
  if (*reinterpret_cast<volatile int*>(abort_flag)) return false;
  if (ptx::mbar_wait(bar, parity, kWaitNs)) return true;
  atomicOr(status, 1u);
  *reinterpret_cast<volatile int*>(abort_flag) = 1;
  return false;
}

// Position of a CTA in its schedule. Work units are (sequence, segment)
// pairs, unit u = seq * nseg + segment, covering chunks [c_begin, c_end) of
// the sequence; a CTA walks units blockIdx.x, +gridDim.x, ... chunk by chunk.
// (32-bit indices, divided once per unit: 64-bit division is a long
// software sequence.)
struct Sched {
  int unit, b, h;
  int c, c_begin, c_end;
  __device__ __forceinline__ void start(int u, const TcParams& p) {
    unit = u;
    const int seq = u / p.nseg;
    c_begin = (u - seq * p.nseg) * p.seg_chunks;
    c_end = min(p.nchunks, c_begin + p.seg_chunks);
    c = c_begin;
    b = seq / p.heads;
    h = seq - b * p.heads;
  }
  __device__ __forceinline__ bool has_next(const TcParams& p) const {
    return c + 1 < c_end || unit + (int)gridDim.x < p.nunits;
  }
  __device__ __forceinline__ bool next(const TcParams& p) {
    if (++c < c_end) return true;
    const int u = unit + (int)gridDim.x;
    if (u >= p.nunits) return false;
    start(u, p);
    return true;
  }
};

// Raw decay inputs of a chunk's tokens: dt, lambda of the token and of its
// successor (zero past the end of the sequence); lane handles tokens lane and
// lane + 32. Only loads, so that their latency overlaps other work.
struct DecayRaw {
  float dt[2], lam[2], dtn[2], lamn[2], A;
};
__device__ __forceinline__ void load_decay_raw(const TcParams& p, const Sched& u, int Q, int lane,
                                               DecayRaw& d) {
  const int64_t L = p.L, H = p.H, b = u.b, h = u.h, t0 = (int64_t)u.c * Q;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int i = lane + 32 * j;
    const int64_t t = t0 + i;
    const bool in = i < Q && t < L, inn = i < Q && t + 1 < L;
    d.dt[j] = in ? p.dt[(b * L + t) * H + h] : 0.f;
    d.lam[j] = in ? p.lam[(b * L + t) * H + h] : 0.f;
    d.dtn[j] = inn ? p.dt[(b * L + t + 1) * H + h] : 0.f;
    d.lamn[j] = inn ? p.lam[(b * L + t + 1) * H + h] : 1.f;
  }
  d.A = p.A[u.h];
}
// The chunk's decay scan (one warp, shuffles): Lam_t = inclusive sum of
// Delta A within the chunk, and the weights derived from it.
__device__ __forceinline__ void decay_scan(const DecayRaw& d, int Q, int lane, Scal& sc) {
  float a0 = d.dt[0] * d.A * kLog2e, a1 = d.dt[1] * d.A * kLog2e;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float v0 = __shfl_up_sync(0xffffffffu, a0, o);
    const float v1 = __shfl_up_sync(0xffffffffu, a1, o);
    if (lane >= o) {
      a0 += v0;
      a1 += v1;
    }
  }
  a1 += __shfl_sync(0xffffffffu, a0, 31);
  const float lam_end = (Q <= 32) ? __shfl_sync(0xffffffffu, a0, Q - 1)
                                  : __shfl_sync(0xffffffffu, a1, (Q - 1) & 31);
  const float lv[2] = {a0, a1};
  float wm = 0.f, wpm = 0.f;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int i = lane + 32 * j;
    if (i < Q) {
      const float gam = d.lam[j] * d.dt[j];
      const float wpv = gam + (1.f - d.lamn[j]) * d.dtn[j];
      wpm = fmaxf(wpm, fmaxf(fabsf(gam), fabsf(wpv)));
      const float we = ex2(lam_end - lv[j]) * wpv;
      sc.lam2[i] = lv[j];
      sc.gam[i] = gam;
      sc.wp[i] = wpv;
      sc.wend[i] = we;
      sc.eL[i] = ex2(lv[j]);
      sc.dt[i] = d.dt[j];
      wm = fmaxf(wm, fabsf(we));
    }
  }
  wm = warp_max(wm);
  wpm = warp_max(wpm);
  if (lane == 0) {
    sc.eLend = ex2(lam_end);
    sc.lamend2 = lam_end;
    sc.wmax = wm;
    sc.wpmax = wpm;
  }
}

// theta of this fold thread's tokens (TPG consecutive tokens of group tg) and
// pairs (k0, k0 + 1), straight from global memory (zero past the end).
template <int KP, int TPG>
__device__ __forceinline__ void load_theta(const TcParams& p, const Sched& u, int Q, int tg, int k0,
                                           float2 (&th)[TPG]) {
  const int64_t gi = u.h / p.hpg;
  const int64_t t0 = (int64_t)u.c * Q + tg * TPG;
#pragma unroll
  for (int i = 0; i < TPG; ++i) {
    const int64_t t = t0 + i;
    th[i] = t < p.L ? __ldg(reinterpret_cast<const float2*>(
                          p.theta + (((int64_t)u.b * p.L + t) * p.G + gi) * KP + k0))
                    : make_float2(0.f, 0.f);
  }
}

// Sum over the KP2 lanes that hold one token row (a whole warp for N = 128,
// a half warp for N = 64).
template <int KP2>
__device__ __forceinline__ float row_sum(float v) {
#pragma unroll
  for (int o = KP2 / 2; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// BCNorm: the inverse root mean square over the N rows of element rank r of
// one token's raw B (or C) words, this thread holding rows 4kk2 .. 4kk2 + 3.
template <int R, int NS, int BW>
__device__ __forceinline__ float bc_inv_rms(const uint32_t (&w)[BW], int r) {
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float v = bf_at(w, e * R + r);
    ss = fmaf(v, v, ss);
  }
  ss = row_sum<NS / 4>(ss);
  return rsqrtf(fmaf(ss, 1.f / NS, 1e-6f));
}

// R = 1, N = 128 (a whole warp holds one token row of B and of C): the
// inverse RMS of V = TPG (B only) or 2 TPG (B, then C) rows at once. A
// reduce-scatter over the lane masks 16, 8, ... leaves each lane the full sum
// of one row (16 shuffles for 16 rows instead of 80), whose inverse RMS is
// then gathered back from the lane holding it.
template <int V>
__device__ __forceinline__ void inv_rms_rows(float (&v)[V], int lane) {
  static_assert(V >= 2 && V <= 16 && (V & (V - 1)) == 0, "a power of two up to 16 rows");
  int m = 16;
#pragma unroll
  for (int n = V; n > 1; n >>= 1, m >>= 1) {
    const bool up = (lane & m) != 0;  // keep the upper half of the rows
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = up ? v[i] : v[i + n / 2];
      const float keep = up ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
  }
#pragma unroll
  for (; m >= 1; m >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], m);
  // lane 32 i / V now holds row i's sum over the warp
  const float r = rsqrtf(fmaf(v[0], 1.f / 128.f, 1e-6f));
#pragma unroll
  for (int i = 0; i < V; ++i) v[i] = __shfl_sync(0xffffffffu, r, i * (32 / V));
}

// SO: the state-only pass of a segmented scan (no C, no outputs).
// NORM: B and C arrive un-normalised; BCNorm them here (each token's and
// rank's vector over N divided by its root mean square), before the bias.
// F32: the fp32 precision mode (see Cfg): one CTA per SM (its tiles take
// about 210 KB of shared memory).
template <int R, int NS, bool SO, bool NORM, bool F32>
__global__ void __launch_bounds__(kThreads, F32 ? 1 : 2)
    scan_tc_kernel(const __grid_constant__ CUtensorMap tm_B, const __grid_constant__ CUtensorMap tm_C,
                   const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_y,
                   TcParams p) {
  using K = Cfg<R, NS, F32>;
  static_assert(!(F32 && NORM), "BCNorm is fused on the bf16 path only");
  constexpr int Q = K::Q, KP = K::KP, KP2 = K::KP2, TG = K::TG, TPG = K::TPG, HR = K::HR;
  constexpr uint32_t kIdS = ptx::idesc_f16_f32(64, 64, false, false);
  constexpr uint32_t kIdD = ptx::idesc_f16_f32(NS, 64, true, true);
  constexpr uint32_t kIdYo = ptx::idesc_f16_f32(64, 64, false, true);
  // Y = P X: fp16 P times the fp16 X operand (F32: their high and low parts)
  constexpr uint32_t kIdY = ptx::idesc_f16_f32(64, 64, false, true);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_addr(smem);

  __shared__ uint64_t bar_raw, bar_ds, bar_yo, bar_y;
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_flag;
  __shared__ Scal ss[2];
  __shared__ __align__(16) float s_tot[TG][KP];  // per token group: angle total
  // F32: its Kahan compensation (the angle sums are compensated in fp32 mode)
  __shared__ __align__(16) float s_totlo[F32 ? TG : 1][F32 ? KP : 2];
  __shared__ float s_carry[2][2][KP];            // [chunk parity][hi, lo][pair]
  __shared__ float s_fang[KP];                   // angle after a unit's last chunk
  __shared__ unsigned int s_max[2][3];  // per chunk parity: bounds of |B|, |C|, |x|
  __shared__ float s_red[kWarps];
  __shared__ float s_red_unit[kWarps];  // the entering state's bound at a unit start
  __shared__ float s_bias_red[2][kWarps];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nC = p.nchunks;
  // fold mapping: pairs k0, k0 + 1 (rows 4kk2 .. 4kk2 + 3), tokens tg*TPG ..
  const int kk2 = tid % KP2, tg = tid / KP2, k0 = 2 * kk2;
  // The next chunk's decay scan: in the full pass by warp 4 during the mask
  // phase (warp 4's 16 rows x 32 columns of S lie above the diagonal for
  // every R, so it only writes zeros there); in the state-only pass by warp 0
  // at the end of the chunk.
  constexpr int kDecayWarp = SO ? 0 : 4;
  // R = 4 (bf16): the raw B, C and x tiles arrive 128-byte swizzled (a thread
  // reads 32 bytes per token row, and unswizzled rows put two lanes of every
  // quarter-warp on the same banks)
  constexpr bool kSwRaw = R == 4 && !F32;
  // The MMAs are issued by lane 0 of warp 5, which (like warp 4) has no share
  // of the mask phase, rather than by thread 0: the issue takes about a
  // microsecond per chunk, which warp 5 spends where it would otherwise wait.
  constexpr int kMmaTid = 160;
  // accumulator mapping: TMEM lane quadrant, 32-column half
  const int quad = warp & 3, half = warp >> 2;

  // ---------------------------------------------------------------- setup
  if (warp == 0) {
    ptx::tmem_alloc(&tmem_holder, kTmemCols);
    ptx::tmem_relinquish();
  }
  if (tid == 0) {
    abort_flag = 0;
    for (int i = 0; i < 6; ++i) (&s_max[0][0])[i] = 0u;
    ptx::mbar_init(&bar_raw, 1);
    ptx::mbar_init(&bar_ds, 1);
    ptx::mbar_init(&bar_yo, 1);
    ptx::mbar_init(&bar_y, 1);
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&tm_B);
    ptx::prefetch_tensormap(&tm_C);
    ptx::prefetch_tensormap(&tm_x);
    if (R > 1) ptx::prefetch_tensormap(&tm_y);
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem = tmem_holder;
  const uint32_t tq = (uint32_t)(32 * quad) << 16;  // this warp's lane quadrant

  // TMA of one chunk's raw tiles into the raw slot (one thread)
  auto issue_raw = [&](const Sched& u) {
    const int gi = u.h / p.hpg;
    const int t0 = u.c * Q;
    ptx::mbar_arrive_expect_tx(&bar_raw, SO ? K::kTxBytesSO : K::kTxBytes);
    ptx::tma_load_5d(smem + K::kRawB, &tm_B, &bar_raw, 0, 0, gi, t0, u.b);
    if (!SO) ptx::tma_load_5d(smem + K::kRawC, &tm_C, &bar_raw, 0, 0, gi, t0, u.b);
    if constexpr (kSwRaw)
      ptx::tma_load_5d(smem + K::kRawX, &tm_x, &bar_raw, 0, 0, u.h, t0, u.b);
    else
      ptx::tma_load_4d(smem + K::kRawX, &tm_x, &bar_raw, 0, u.h, t0, u.b);
  };

  // state element (n, cb + j) of this thread's 16-column block `blk` is hv[16 blk + j]
  auto hpos = [&](int blk, uint32_t& n, uint32_t& cb) {
    if constexpr (NS == 128) {
      n = (uint32_t)(32 * quad + lane);  // M=128 accumulator layout: lane = row
      cb = 32u * half + 16u * blk;
    } else {
      n = (uint32_t)(16 * quad + (lane & 15));  // M=64 layout: 16 rows per quadrant
      cb = 32u * half + 16u * (lane >> 4);
    }
  };
  auto state_ld = [&](float (&hv)[HR]) {
#pragma unroll
    for (int blk = 0; blk < HR / 16; ++blk) {
      uint32_t d[16];
      if constexpr (NS == 128)
        ptx::tmem_ld16(tmem + kColD + tq + 32u * half + 16u * blk, d);
      else
        ptx::tmem_ld16_16x32bx2<16>(tmem + kColD + tq + 32u * half, d);
      ptx::tmem_ld_wait(d);
#pragma unroll
      for (int j = 0; j < 16; ++j) hv[16 * blk + j] = __uint_as_float(d[j]);
    }
  };
  auto state_st = [&](const float (&hv)[HR]) {
#pragma unroll
    for (int blk = 0; blk < HR / 16; ++blk) {
      uint32_t d[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) d[j] = __float_as_uint(hv[16 * blk + j]);
      if constexpr (NS == 128)
        ptx::tmem_st16(tmem + kColD + tq + 32u * half + 16u * blk, d);
      else
        ptx::tmem_st16_16x32bx2<16>(tmem + kColD + tq + 32u * half, d);
    }
    ptx::tmem_st_wait();
  };
  // fp16 copy of f * hv into the state tile (operand of the next Yoff)
  auto write_hcopy = [&](const float (&hv)[HR], float f) {
    const float2 f2 = make_float2(f, f);
#pragma unroll
    for (int blk = 0; blk < HR / 16; ++blk) {
      uint32_t n, cb;
      hpos(blk, n, cb);
      uint32_t wv[8], wl[8];
#pragma unroll
      for (int j = 0; j < 16; j += 2) {
        const float2 v = mul2(f2, make_float2(hv[16 * blk + j], hv[16 * blk + j + 1]));
        wv[j >> 1] = pack_f16(v.x, v.y);
        if constexpr (F32) wl[j >> 1] = f16_residual(wv[j >> 1], v.x, v.y);
      }
      sts128(sbase + K::kH + sw128(n, cb), make_uint4(wv[0], wv[1], wv[2], wv[3]));
      sts128(sbase + K::kH + sw128(n, cb + 8u), make_uint4(wv[4], wv[5], wv[6], wv[7]));
      if constexpr (F32) {
        sts128(sbase + K::kH + K::kHLo + sw128(n, cb), make_uint4(wl[0], wl[1], wl[2], wl[3]));
        sts128(sbase + K::kH + K::kHLo + sw128(n, cb + 8u), make_uint4(wl[4], wl[5], wl[6], wl[7]));
      }
    }
  };
  auto abs_max = [&](const float (&hv)[HR]) {
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < HR; ++i) m = fmaxf(m, fabsf(hv[i]));
    return m;
  };

  // Fold stores: row l = i R + r of this thread's token rows (rows tg*TPG*R +
  // l) at columns 4kk2 .. 4kk2 + 3 of Bt / Ct. The 128-byte swizzle XORs the
  // 16-byte chunk index with the row's low three bits; those are rb7 ^ (l & 7)
  // (rb7 = the first row's, 0 or 4), so every store address is the one base
  // below XOR (l & 7) << 4 (bits 4-6, which nothing else in the base sets)
  // plus the constant l * 128.
  uint32_t fold_base;
  {
    const uint32_t col = 4u * (uint32_t)kk2, cl = col & 63u;
    const uint32_t row0 = (uint32_t)(tg * TPG * R), rb7 = row0 & 7u;
    fold_base = sbase + K::kBt + (col >> 6) * 64u * 128u + row0 * 128u +
                ((((cl >> 3) ^ rb7) & 7u) << 4) + (cl & 7u) * 2u;
  }

  // ---------------------------------------------------------------- first chunk's inputs
  Sched sch;
  sch.start(blockIdx.x, p);
  if (tid == 0) issue_raw(sch);
  DecayRaw dr;
  if (warp == kDecayWarp) {
    load_decay_raw(p, sch, Q, lane, dr);
    decay_scan(dr, Q, lane, ss[0]);
  }
  float2 th[TPG];
  load_theta<KP, TPG>(p, sch, Q, tg, k0, th);
  __syncthreads();

  // state bookkeeping (uniform over the CTA)
  bool has_state = false;   // TMEM holds a state (else the first D MMA overwrites)
  bool yoff_ready = false;  // the state tile holds H_in of this chunk (its Yoff is issued)
  float u_prev = 1.f;       // the TMEM state is (state) / u_prev
  float h_inv_prev = 1.f;   // inverse scale of the state tile read by this chunk's Yoff
  float dsum = 0.f;         // log2 decay over the unit (state-only pass)
  float bmax_bias = 0.f, cmax_bias = 0.f;  // bounds of the head's bias magnitudes
  // (thread 0) parity of a raw load issued and not yet waited for; (the MMA
  // thread) the barrier and parity of its last commit: what an early exit
  // waits for
  int raw_pending = 0;
  uint64_t* last_commit = nullptr;
  uint32_t last_parity = 0;
  float hv[HR];

  for (int g = 0;; ++g) {
    const int b = sch.b, h = sch.h, c = sch.c;
    const bool first = c == sch.c_begin, last = c == sch.c_end - 1;
    const bool has_next = sch.has_next(p);
    Scal& sc = ss[g & 1];
    ptx::tc_fence_after_sync();

    // ================================================= unit start: entering state
    if (first) {
      has_state = false;
      yoff_ready = false;
      u_prev = 1.f;
      dsum = 0.f;
      {
        // bounds of the head's bias magnitudes (for the fp16 scales)
        const int64_t o = ((int64_t)h * NS + 4 * kk2) * R;
        float bm = 0.f, cm = 0.f;
#pragma unroll
        for (int q = 0; q < R; ++q) {
          const float4 vb = p.B_bias ? __ldg(reinterpret_cast<const float4*>(p.B_bias + o) + q)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
          const float4 vc = (!SO && p.C_bias)
                                ? __ldg(reinterpret_cast<const float4*>(p.C_bias + o) + q)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
          bm = fmaxf(bm, fmaxf(fmaxf(fabsf(vb.x), fabsf(vb.y)), fmaxf(fabsf(vb.z), fabsf(vb.w))));
          cm = fmaxf(cm, fmaxf(fmaxf(fabsf(vc.x), fabsf(vc.y)), fmaxf(fabsf(vc.z), fabsf(vc.w))));
        }
        bm = warp_max(bm);
        cm = warp_max(cm);
        if (lane == 0) {
          s_bias_red[0][warp] = bm;
          s_bias_red[1][warp] = cm;
        }
        __syncthreads();
        bmax_bias = 0.f;
        cmax_bias = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          bmax_bias = fmaxf(bmax_bias, s_bias_red[0][w]);
          cmax_bias = fmaxf(cmax_bias, s_bias_red[1][w]);
        }
      }
      if (p.ws_hin) {
        // the given explicit-frame state (the unit's angle frame starts at
        // zero, so no rotation) goes into TMEM as it is; the full pass also
        // writes its fp16 copy for the first chunk's Yoff
        const float* src = p.ws_hin + (int64_t)sch.unit * NS * kP;
#pragma unroll
        for (int blk = 0; blk < HR / 16; ++blk) {
          uint32_t n, cb;
          hpos(blk, n, cb);
          const float4* q4 = reinterpret_cast<const float4*>(src + (int64_t)n * kP + cb);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float4 v = q4[j];
            hv[16 * blk + 4 * j] = v.x;
            hv[16 * blk + 4 * j + 1] = v.y;
            hv[16 * blk + 4 * j + 2] = v.z;
            hv[16 * blk + 4 * j + 3] = v.w;
          }
        }
        state_st(hv);
        has_state = true;
        if constexpr (!SO) {
          const float m = warp_max(abs_max(hv));
          if (lane == 0) s_red_unit[warp] = m;
          __syncthreads();
          float mm = 0.f;
#pragma unroll
          for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, s_red_unit[w]);
          float h_sig;
          pow2_scale(mm, &h_sig, &h_inv_prev);
          write_hcopy(hv, h_sig);
          yoff_ready = true;
          // the block barrier before the MMA issue orders these writes
        }
      }
    }

    // ================================================= fold, part 1
    Sched nxt = sch;
    if (has_next) nxt.next(p);
    // state-only pass: warp 0's loads of the next chunk's decay inputs (used
    // at the end of this chunk), a whole fold ahead of their use
    if (SO && warp == kDecayWarp && has_next) load_decay_raw(p, nxt, Q, lane, dr);
    // every thread waits for this chunk's raw tiles itself
    if (wait_or_abort(&bar_raw, (uint32_t)(g & 1), &abort_flag, p.status) && tid == 0)
      raw_pending = -1;
    // raw B, C tiles -> registers
    uint32_t bw[TPG][K::BW], cw[TPG][K::BW];
    uint32_t bacc = 0u, cacc = 0u;
    float bfm = 0.f, cfm = 0.f;  // F32: magnitude bounds
#pragma unroll
    for (int i = 0; i < TPG; ++i) {
      const int t = tg * TPG + i;
      const uint32_t ob = (uint32_t)(t * NS * R + 4 * kk2 * R) * (uint32_t)K::AB;
      if constexpr (F32) {
#pragma unroll
        for (int q = 0; q < K::BW / 4; ++q) {
          const uint4 vb = lds128(sbase + K::kRawB + ob + 16u * q);
          bw[i][4 * q] = vb.x; bw[i][4 * q + 1] = vb.y; bw[i][4 * q + 2] = vb.z; bw[i][4 * q + 3] = vb.w;
          if constexpr (!SO) {
            const uint4 vc = lds128(sbase + K::kRawC + ob + 16u * q);
            cw[i][4 * q] = vc.x; cw[i][4 * q + 1] = vc.y; cw[i][4 * q + 2] = vc.z; cw[i][4 * q + 3] = vc.w;
          }
        }
      } else if constexpr (R == 1) {
        const uint2 vb = lds64(sbase + K::kRawB + ob);
        bw[i][0] = vb.x;
        bw[i][1] = vb.y;
        if constexpr (!SO) {
          const uint2 vc = lds64(sbase + K::kRawC + ob);
          cw[i][0] = vc.x;
          cw[i][1] = vc.y;
        }
      } else {
#pragma unroll
        for (int q = 0; q < K::BW / 4; ++q) {
          uint32_t o = ob + 16u * q;
          if constexpr (kSwRaw) {
            // token t's NS / 16 rows of 128 bytes; this thread's 32 bytes are
            // chunks 2 (kk2 & 3) + q of row t NS / 16 + kk2 / 4
            const uint32_t row = (uint32_t)(t * (NS / 16) + kk2 / 4);
            o = row * 128u + ((((uint32_t)(2 * (kk2 & 3) + q)) ^ (row & 7u)) << 4);
          }
          const uint4 vb = lds128(sbase + K::kRawB + o);
          bw[i][4 * q] = vb.x; bw[i][4 * q + 1] = vb.y; bw[i][4 * q + 2] = vb.z; bw[i][4 * q + 3] = vb.w;
          if constexpr (!SO) {
            const uint4 vc = lds128(sbase + K::kRawC + o);
            cw[i][4 * q] = vc.x; cw[i][4 * q + 1] = vc.y; cw[i][4 * q + 2] = vc.z; cw[i][4 * q + 3] = vc.w;
          }
        }
      }
    }
    if constexpr (F32) {
#pragma unroll
      for (int i = 0; i < TPG; ++i) {
#pragma unroll
        for (int q = 0; q < K::BW; ++q) {
          bfm = fmaxf(bfm, fabsf(__uint_as_float(bw[i][q])));
          if constexpr (!SO) cfm = fmaxf(cfm, fabsf(__uint_as_float(cw[i][q])));
        }
      }
    } else if constexpr (!NORM) {
#pragma unroll
      for (int i = 0; i < TPG; ++i) {
#pragma unroll
        for (int q = 0; q < K::BW; ++q) {
          bacc = ptx::bf16x2_absmax(bacc, bw[i][q]);
          if constexpr (!SO) cacc = ptx::bf16x2_absmax(cacc, cw[i][q]);
        }
      }
    }
    // x of this chunk -> registers (w X and the operand copy of X). An item
    // is 8 consecutive p of one token row (R = 1; bf16: the 16-byte chunk at
    // the same place of the 128B-swizzled raw tile) or 4 p x R ranks (R > 1).
    constexpr int kXItems = (R == 1) ? 2 : (Q * (kP / 4)) / kThreads;
    uint32_t xw[kXItems][K::XW];
    uint32_t xacc = 0u;
    float xfm = 0.f;
#pragma unroll
    for (int j = 0; j < kXItems; ++j) {
      const int it = tid + kThreads * j;
      uint32_t src;
      if constexpr (R == 1) {
        src = F32 ? sbase + K::kRawX + (uint32_t)it * 32u   // fp32 row-major: 8 floats
                  : sbase + K::kRawX + (uint32_t)it * 16u;  // physical 16-byte chunk
      } else {
        const int sx = it / (kP / 4), pb = it % (kP / 4);
        src = sbase + K::kRawX + (uint32_t)(sx * kP * R + 4 * pb * R) * (uint32_t)K::AB;
      }
#pragma unroll
      for (int q = 0; q < K::XW / 4; ++q) {
        uint32_t a_ = src + 16u * q;
        if constexpr (kSwRaw) {
          // token sx's four rows of 128 bytes (64 (p, r) elements each)
          const int sx = it / (kP / 4), pb = it % (kP / 4);
          const uint32_t row = (uint32_t)(sx * 4 + pb / 4);
          a_ = sbase + K::kRawX + row * 128u + ((((uint32_t)(2 * (pb & 3) + q)) ^ (row & 7u)) << 4);
        }
        const uint4 v = lds128(a_);
        xw[j][4 * q] = v.x; xw[j][4 * q + 1] = v.y; xw[j][4 * q + 2] = v.z; xw[j][4 * q + 3] = v.w;
      }
#pragma unroll
      for (int q = 0; q < K::XW; ++q) {
        if constexpr (F32)
          xfm = fmaxf(xfm, fabsf(__uint_as_float(xw[j][q])));
        else
          xacc = ptx::bf16x2_absmax(xacc, xw[j][q]);
      }
    }
    // per-token-group angle sums (pairs k0, k0 + 1)
    float2 ph[TPG];
    {
      float2 run = make_float2(0.f, 0.f), comp = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < TPG; ++i) {
        const float d = sc.dt[tg * TPG + i];
        if constexpr (F32) {
          // Kahan-compensated: the fp32 mode's angles stay exact to ~2^-24
          const float2 yk = ptx::sub2(mul2(make_float2(d, d), th[i]), comp);
          const float2 tk = add2(run, yk);
          comp = ptx::sub2(ptx::sub2(tk, run), yk);
          run = tk;
        } else {
          run = fma2(make_float2(d, d), th[i], run);
        }
        ph[i] = run;
      }
      *reinterpret_cast<float2*>(&s_tot[tg][k0]) = run;
      if constexpr (F32)
        *reinterpret_cast<float2*>(&s_totlo[tg][k0]) = make_float2(-comp.x, -comp.y);
    }
    {
      // non-negative floats order like their bit patterns
      const float bm = warp_max(F32 ? bfm : bf_absmax(bacc));
      const float cm = warp_max(F32 ? cfm : bf_absmax(cacc));
      const float xm = warp_max(F32 ? xfm : bf_absmax(xacc));
      if (lane == 0) {
        atomicMax(&s_max[g & 1][0], __float_as_uint(bm));
        atomicMax(&s_max[g & 1][1], __float_as_uint(cm));
        atomicMax(&s_max[g & 1][2], __float_as_uint(xm));
      }
    }
    // the staging tile of the previous chunk's output (over w X) is free
    if (!SO && R > 1 && tid == 0) ptx::tma_store_wait_read<0>();
    __syncthreads();  // ------------------------------------------ fold A
    if (*reinterpret_cast<volatile int*>(&abort_flag)) break;
    ptx::tc_fence_after_sync();
    // every read of the raw slot is done: refill it with the next chunk
    if (has_next && tid == 0) {
      issue_raw(nxt);
      raw_pending = (g + 1) & 1;
    }

    // ================================================= fold, part 2
    float sigB, invB, sigC, invC, sigX, invX;
    float sigXo = 1.f;  // scale of the X operand tile
    {
      const float mb = __uint_as_float(s_max[g & 1][0]);
      const float mc = __uint_as_float(s_max[g & 1][1]);
      const float mx = __uint_as_float(s_max[g & 1][2]);
      // the other parity's words were read last chunk: clear them for the next
      if (tid == 0) {
#pragma unroll
        for (int i = 0; i < 3; ++i) s_max[(g + 1) & 1][i] = 0u;
      }
      // a rotated pair keeps its norm: |Rot(v)_i| <= sqrt(2) max|v| < 2 max|v|;
      // a BCNormed vector has every element below sqrt(N) in magnitude
      constexpr float kNormBound = (NS == 128) ? 11.3137085f : 8.f;
      // The state in TMEM is held in units of sigma_B sigma_X (the D MMA's):
      // the tile scales are capped at 2^40, so that a chunk of zero or tiny
      // inputs after large ones cannot inflate it beyond fp32's range (with
      // the cap, elements above 2^-54 still keep fp16's full precision).
      pow2_scale<-26>(2.f * ((NORM ? kNormBound : mb) + bmax_bias), &sigB, &invB);
      pow2_scale<-26>(2.f * ((NORM ? kNormBound : mc) + cmax_bias), &sigC, &invC);
      pow2_scale<-26>(mx * sc.wmax, &sigX, &invX);
      float pmul = invB * invC;
      {
        // the X operand (fp16; F32: hi + lo) by its own scale; P by one from
        // a bound of |P|: |S| <= N max|Bt| max|Ct|, the mask <= max(|gamma|,
        // |gamma + bhat|)
        float invXo, sigP, invP;
        pow2_scale(mx, &sigXo, &invXo);
        pow2_scale((float)NS * (2.f * ((NORM ? kNormBound : mb) + bmax_bias)) *
                       (2.f * ((NORM ? kNormBound : mc) + cmax_bias)) * sc.wpmax,
                   &sigP, &invP);
        pmul *= sigP;
        if (tid == 0) sc.ykY = invP * invXo;
      }
      if (tid == 0) {
        sc.invB = invB;
        sc.invC = invC;
        sc.invX = invX;
        sc.pmul = pmul;
      }
    }
    // angle before this thread's first token: carry + earlier groups. Within
    // the chunk an fp32 offset suffices; the carry to the next chunk is
    // float-float so that it does not drift.
    const int cpar = g & 1;
    {
      float2 o = make_float2(0.f, 0.f);
#pragma unroll
      for (int q = 0; q < TG - 1; ++q) {
        float2 v = *reinterpret_cast<const float2*>(&s_tot[q][k0]);
        if constexpr (F32) v = add2(v, *reinterpret_cast<const float2*>(&s_totlo[q][k0]));
        if (q < tg) o = add2(o, v);
      }
      float ch0 = 0.f, cl0 = 0.f, ch1 = 0.f, cl1 = 0.f;
      if (!first) {
        ch0 = s_carry[cpar][0][k0];
        cl0 = s_carry[cpar][1][k0];
        ch1 = s_carry[cpar][0][k0 + 1];
        cl1 = s_carry[cpar][1][k0 + 1];
      }
      const float2 off = make_float2(wrap_rad(ch0 + (cl0 + o.x)), wrap_rad(ch1 + (cl1 + o.y)));
      // the carry of pair k0 is updated by group TG-1, that of k0+1 by TG-2
      if (tg >= TG - 2) {
        const int k = (tg == TG - 1) ? k0 : k0 + 1;
        // float-float sum of the group totals as a tree, then the carry
        float thh[TG], tll[TG];
#pragma unroll
        for (int q = 0; q < TG; ++q) {
          thh[q] = s_tot[q][k];
          tll[q] = F32 ? s_totlo[q][k] : 0.f;
        }
#pragma unroll
        for (int w = 1; w < TG; w <<= 1)
#pragma unroll
          for (int q = 0; q + w < TG; q += 2 * w) ff_add(thh[q], tll[q], thh[q + w], tll[q + w]);
        float eh = (tg == TG - 1) ? ch0 : ch1, el = (tg == TG - 1) ? cl0 : cl1;
        ff_add(eh, el, thh[0], tll[0]);
        ff_wrap(eh, el);
        s_carry[cpar ^ 1][0][k] = eh;
        s_carry[cpar ^ 1][1][k] = el;
        if (last) s_fang[k] = eh + el;
      }
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < TPG; ++i) {
        ph[i] = add2(off, ph[i]);
        amax = fmaxf(amax, fmaxf(fabsf(ph[i].x), fabsf(ph[i].y)));
      }
      // (the fp32 mode always reduces: sin.approx / cos.approx are exact to
      // ~2^-21 in absolute terms only on [-pi, pi])
      if (F32 || __any_sync(0xffffffffu, amax > kAngleDirect)) {
#pragma unroll
        for (int i = 0; i < TPG; ++i) ph[i] = make_float2(wrap_rad(ph[i].x), wrap_rad(ph[i].y));
      }
    }
    // w X (fp16, scaled) and X as the [(token, rank)][p] operand: fp16 of
    // sigXo x (exact for bf16 inputs), or (F32) its fp16 hi + lo
#pragma unroll
    for (int j = 0; j < kXItems; ++j) {
      const int it = tid + kThreads * j;
      if constexpr (R == 1 && !F32) {
        // the raw tile is already 128-byte swizzled [token][p]: same offsets
        const uint32_t row = (uint32_t)it >> 3;
        const float w = sc.wend[row] * sigX;
        const float2 w2 = make_float2(w, w);
        const float2 x0 = make_float2(bf_lo(xw[j][0]), bf_hi(xw[j][0]));
        const float2 x1 = make_float2(bf_lo(xw[j][1]), bf_hi(xw[j][1]));
        const float2 x2 = make_float2(bf_lo(xw[j][2]), bf_hi(xw[j][2]));
        const float2 x3 = make_float2(bf_lo(xw[j][3]), bf_hi(xw[j][3]));
        if constexpr (!SO) {
          const float2 s2 = make_float2(sigXo, sigXo);
          const float2 q0 = mul2(s2, x0), q1 = mul2(s2, x1), q2 = mul2(s2, x2), q3 = mul2(s2, x3);
          sts128(sbase + K::kXo + (uint32_t)it * 16u,
                 make_uint4(pack_f16(q0.x, q0.y), pack_f16(q1.x, q1.y), pack_f16(q2.x, q2.y),
                            pack_f16(q3.x, q3.y)));
        }
        const float2 p0 = mul2(w2, x0), p1 = mul2(w2, x1), p2 = mul2(w2, x2), p3 = mul2(w2, x3);
        sts128(sbase + K::kXw + (uint32_t)it * 16u,
               make_uint4(pack_f16(p0.x, p0.y), pack_f16(p1.x, p1.y), pack_f16(p2.x, p2.y),
                          pack_f16(p3.x, p3.y)));
      } else if constexpr (R == 1) {
        // F32: item it holds p = 8 (it & 7) .. + 7 of row it / 8 (row-major raw)
        const uint32_t row = (uint32_t)it >> 3;
        const float w = sc.wend[row] * sigX;
        const float2 w2 = make_float2(w, w);
        const uint32_t o = sw128(row, 8u * ((uint32_t)it & 7u));
        uint32_t hw[4], hl[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const float2 pw = mul2(w2, make_float2(act_at<F32>(xw[j], e), act_at<F32>(xw[j], e + 1)));
          hw[e >> 1] = pack_f16(pw.x, pw.y);
          hl[e >> 1] = f16_residual(hw[e >> 1], pw.x, pw.y);
        }
        sts128(sbase + K::kXw + o, make_uint4(hw[0], hw[1], hw[2], hw[3]));
        sts128(sbase + K::kXw + K::kXLo + o, make_uint4(hl[0], hl[1], hl[2], hl[3]));
        if constexpr (!SO) {
          const float2 s2 = make_float2(sigXo, sigXo);
          uint32_t ph4[4], pl4[4];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const float2 px = mul2(s2, make_float2(act_at<F32>(xw[j], e), act_at<F32>(xw[j], e + 1)));
            ph4[e >> 1] = pack_f16(px.x, px.y);
            pl4[e >> 1] = f16_residual(ph4[e >> 1], px.x, px.y);
          }
          sts128(sbase + K::kXo + o, make_uint4(ph4[0], ph4[1], ph4[2], ph4[3]));
          sts128(sbase + K::kXo + K::kXLo + o, make_uint4(pl4[0], pl4[1], pl4[2], pl4[3]));
        }
      } else {
        const int sx = it / (kP / 4), pb = it % (kP / 4);
        const float w = sc.wend[sx] * sigX;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          float v4[4];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) v4[q4] = act_at<F32>(xw[j], q4 * R + r);
          const uint32_t o = sw128((uint32_t)(sx * R + r), 4u * pb);
          const uint32_t w0 = pack_f16(w * v4[0], w * v4[1]), w1 = pack_f16(w * v4[2], w * v4[3]);
          sts64(sbase + K::kXw + o, w0, w1);
          if constexpr (F32) {
            sts64(sbase + K::kXw + K::kXLo + o, f16_residual(w0, w * v4[0], w * v4[1]),
                  f16_residual(w1, w * v4[2], w * v4[3]));
            if constexpr (!SO) {
              const float a0 = sigXo * v4[0], a1 = sigXo * v4[1], a2 = sigXo * v4[2],
                          a3 = sigXo * v4[3];
              const uint32_t x0 = pack_f16(a0, a1), x1 = pack_f16(a2, a3);
              sts64(sbase + K::kXo + o, x0, x1);
              sts64(sbase + K::kXo + K::kXLo + o, f16_residual(x0, a0, a1), f16_residual(x1, a2, a3));
            }
          } else if constexpr (!SO) {
            sts64(sbase + K::kXo + o, pack_f16(sigXo * v4[0], sigXo * v4[1]),
                  pack_f16(sigXo * v4[2], sigXo * v4[3]));
          }
        }
      }
    }
    // RoPE fold: sigma Rot(-Phi) (B + bias), likewise C, into fp16 tiles
    const uint32_t opBt = sbase + K::kBt, opCt = sbase + K::kCt;
    const float2 sB2 = make_float2(sigB, sigB), sC2 = make_float2(sigC, sigC);
    if constexpr (R == 1) {
      // sigma (B + bias) = fma(sigma, B, sigma bias), exact for a power-of-two
      // sigma, so the scale rides on the bias add instead of on cos and sin
      const int64_t ob = (int64_t)h * NS + 4 * kk2;
      float4 bq[1], cq[1];
      bq[0] = p.B_bias ? __ldg(reinterpret_cast<const float4*>(p.B_bias + ob))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      cq[0] = (!SO && p.C_bias) ? __ldg(reinterpret_cast<const float4*>(p.C_bias + ob))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
      const float2 bs0 = mul2(sB2, make_float2(bq[0].x, bq[0].z));
      const float2 bs1 = mul2(sB2, make_float2(bq[0].y, bq[0].w));
      const float2 cs0 = mul2(sC2, make_float2(cq[0].x, cq[0].z));
      const float2 cs1 = mul2(sC2, make_float2(cq[0].y, cq[0].w));
      // (NORM, N = 128) the tokens' inverse RMS of B, then of C, all at once
      constexpr bool kRowsAtOnce = NORM && NS == 128;
      constexpr int kNR = kRowsAtOnce ? (SO ? TPG : 2 * TPG) : 2;
      float irs[kNR];
      if constexpr (kRowsAtOnce) {
#pragma unroll
        for (int i = 0; i < TPG; ++i) {
          float sb = 0.f, sc2 = 0.f;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float vb = bf_at(bw[i], e);
            sb = fmaf(vb, vb, sb);
            if constexpr (!SO) {
              const float vc = bf_at(cw[i], e);
              sc2 = fmaf(vc, vc, sc2);
            }
          }
          irs[i] = sb;
          if constexpr (!SO) irs[TPG + i] = sc2;
        }
        inv_rms_rows<kNR>(irs, lane);
      }
#pragma unroll
      for (int i = 0; i < TPG; ++i) {
        float2 sn, cs;
        __sincosf(ph[i].x, &sn.x, &cs.x);
        __sincosf(ph[i].y, &sn.y, &cs.y);
        const float2 nsn = make_float2(-sn.x, -sn.y);
        // .x holds pair k0 (rows 4kk2, 4kk2 + 1), .y pair k0 + 1
        float2 sBi = sB2;
        if constexpr (NORM) {
          const float v = sigB * (kRowsAtOnce ? irs[i] : bc_inv_rms<R, NS, K::BW>(bw[i], 0));
          sBi = make_float2(v, v);
        }
        const float2 b0 = fma2(sBi, make_float2(act_at<F32>(bw[i], 0), act_at<F32>(bw[i], 2)), bs0);
        const float2 b1 = fma2(sBi, make_float2(act_at<F32>(bw[i], 1), act_at<F32>(bw[i], 3)), bs1);
        // Rot(-Phi) = [[cos, sin], [-sin, cos]]
        const float2 bt0 = fma2(cs, b0, mul2(sn, b1)), bt1 = fma2(cs, b1, mul2(nsn, b0));
        const uint32_t a = (fold_base ^ ((uint32_t)(i & 7) << 4)) + (uint32_t)i * 128u;
        {
          const uint32_t h0 = pack_f16(bt0.x, bt1.x), h1 = pack_f16(bt0.y, bt1.y);
          sts64(a, h0, h1);
          if constexpr (F32)
            sts64(a + K::kBtLo, f16_residual(h0, bt0.x, bt1.x), f16_residual(h1, bt0.y, bt1.y));
        }
        if constexpr (!SO) {
          float2 sCi = sC2;
          if constexpr (NORM) {
            const float v =
                sigC * (kRowsAtOnce ? irs[(TPG + i) % kNR] : bc_inv_rms<R, NS, K::BW>(cw[i], 0));
            sCi = make_float2(v, v);
          }
          const float2 c0 = fma2(sCi, make_float2(act_at<F32>(cw[i], 0), act_at<F32>(cw[i], 2)), cs0);
          const float2 c1 = fma2(sCi, make_float2(act_at<F32>(cw[i], 1), act_at<F32>(cw[i], 3)), cs1);
          const float2 ct0 = fma2(cs, c0, mul2(sn, c1)), ct1 = fma2(cs, c1, mul2(nsn, c0));
          const uint32_t h0 = pack_f16(ct0.x, ct1.x), h1 = pack_f16(ct0.y, ct1.y);
          sts64(a + (K::kCt - K::kBt), h0, h1);
          if constexpr (F32)
            sts64(a + (K::kCt - K::kBt) + K::kBtLo, f16_residual(h0, ct0.x, ct1.x),
                  f16_residual(h1, ct0.y, ct1.y));
        }
      }
    } else {
      // R > 1: B, then C (one bias run live at a time). The thread's rows
      // 4kk2 + e carry the head's bias [n][r]: float4 e holds row 4kk2 + e's R
      // ranks (R = 4; for R = 2 a float4 holds two rows).
      float2 csv[TPG], snv[TPG];
#pragma unroll
      for (int i = 0; i < TPG; ++i) {
        __sincosf(ph[i].x, &snv[i].x, &csv[i].x);
        __sincosf(ph[i].y, &snv[i].y, &csv[i].y);
      }
      const int64_t ob = ((int64_t)h * NS + 4 * kk2) * R;
      // (NORM, N = 128) the inverse RMS of every (token, rank) row of B, then
      // of C, all at once: row (i, r) of pass q is entry (q TPG + i) R + r
      constexpr bool kRowsAtOnce = NORM && NS == 128;
      constexpr int kNR = kRowsAtOnce ? (SO ? 1 : 2) * TPG * R : 2;
      float irs[kNR];
      if constexpr (kRowsAtOnce) {
#pragma unroll
        for (int q = 0; q < (SO ? 1 : 2); ++q)
#pragma unroll
          for (int i = 0; i < TPG; ++i)
#pragma unroll
            for (int r = 0; r < R; ++r) {
              float ss = 0.f;
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float v = bf_at(q == 0 ? bw[i] : cw[i], e * R + r);
                ss = fmaf(v, v, ss);
              }
              irs[(q * TPG + i) * R + r] = ss;
            }
        inv_rms_rows<kNR>(irs, lane);
      }
#pragma unroll
      for (int pass = 0; pass < (SO ? 1 : 2); ++pass) {
        const float* bias = pass == 0 ? p.B_bias : p.C_bias;
        const uint32_t(&raw)[TPG][K::BW] = pass == 0 ? bw : cw;
        const float2 s2 = pass == 0 ? sB2 : sC2;
        float bv[4 * R];
#pragma unroll
        for (int q = 0; q < R; ++q) {
          const float4 v = bias ? __ldg(reinterpret_cast<const float4*>(bias + ob) + q)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
          bv[4 * q] = v.x; bv[4 * q + 1] = v.y; bv[4 * q + 2] = v.z; bv[4 * q + 3] = v.w;
        }
        float2 cs[TPG], sn[TPG], nsn[TPG];
#pragma unroll
        for (int i = 0; i < TPG; ++i) {
          cs[i] = mul2(csv[i], s2);
          sn[i] = mul2(snv[i], s2);
          nsn[i] = make_float2(-sn[i].x, -sn[i].y);
        }
        const uint32_t dst = fold_base + (pass == 0 ? 0u : K::kCt - K::kBt);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          // bias of rows 4kk2 + e, rank r: element e * R + r of the run
          const float2 bb0 = make_float2(bv[0 * R + r], bv[2 * R + r]);
          const float2 bb1 = make_float2(bv[1 * R + r], bv[3 * R + r]);
#pragma unroll
          for (int i = 0; i < TPG; ++i) {
            const float2 v0 = make_float2(act_at<F32>(raw[i], 0 * R + r), act_at<F32>(raw[i], 2 * R + r));
            const float2 v1 = make_float2(act_at<F32>(raw[i], 1 * R + r), act_at<F32>(raw[i], 3 * R + r));
            float2 b0, b1;
            if constexpr (NORM) {
              const float rs = kRowsAtOnce ? irs[((pass * TPG + i) * R + r) % kNR]
                                           : bc_inv_rms<R, NS, K::BW>(raw[i], r);
              b0 = fma2(make_float2(rs, rs), v0, bb0);
              b1 = fma2(make_float2(rs, rs), v1, bb1);
            } else {
              b0 = add2(v0, bb0);
              b1 = add2(v1, bb1);
            }
            const float2 t0 = fma2(cs[i], b0, mul2(sn[i], b1));
            const float2 t1 = fma2(cs[i], b1, mul2(nsn[i], b0));
            const int l = i * R + r;
            const uint32_t a = (dst ^ ((uint32_t)(l & 7) << 4)) + (uint32_t)l * 128u;
            const uint32_t h0 = pack_f16(t0.x, t1.x), h1 = pack_f16(t0.y, t1.y);
            sts64(a, h0, h1);
            if constexpr (F32)
              sts64(a + K::kBtLo, f16_residual(h0, t0.x, t1.x), f16_residual(h1, t0.y, t1.y));
          }
        }
      }
    }
    // the state in TMEM: rescale by exp(Lam_end) and the change of scale, so
    // that D (in units of 1 / (sigma_B sigma_X)) accumulates onto it
    if (has_state) {
      if constexpr (SO) {
        // the previous chunk's D must be complete (in the full pass the
        // previous chunk's mask phase waited for it)
        if (g > 0) wait_or_abort(&bar_ds, (uint32_t)((g - 1) & 1), &abort_flag, p.status);
        ptx::tc_fence_after_sync();
      }
      state_ld(hv);
      const float f = sc.eLend * (sigB * sigX) * u_prev;
      const float2 f2 = make_float2(f, f);
#pragma unroll
      for (int i = 0; i < HR; i += 2) {
        const float2 v = mul2(f2, make_float2(hv[i], hv[i + 1]));
        hv[i] = v.x;
        hv[i + 1] = v.y;
      }
      state_st(hv);
    }
    u_prev = invB * invX;
    // the next chunk's theta and decay inputs (loads only; used next chunk).
    // The full pass issues them after the fold barrier, while the MMAs run,
    // so that no warp reaches that barrier late behind its loads.
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before_sync();
    __syncthreads();  // ------------------------------------------ fold B
    if (*reinterpret_cast<volatile int*>(&abort_flag)) break;
    if (tid == kMmaTid) {
      // D = Bt^T (w X) onto the state; S = Ct Bt^T; Yoff = Ct H_in
      // (F32: every product is hi hi + hi lo + lo hi of the split operands)
      ptx::tc_fence_after_sync();
      const Desc dBm = make_desc(opBt, 64u * 128u), dXw = make_desc(sbase + K::kXw, 64u * 128u);
#pragma unroll
      for (int kk = 0; kk < kQR / 16; ++kk) {
        ptx::mma_f16_ss(tmem + kColD, desc_at(dBm, koff_mn(kk)), desc_at(dXw, koff_mn(kk)), kIdD,
                         (has_state || kk > 0) ? 1u : 0u);
        if constexpr (F32) {
          const Desc dBml = make_desc(opBt + K::kBtLo, 64u * 128u);
          const Desc dXwl = make_desc(sbase + K::kXw + K::kXLo, 64u * 128u);
          ptx::mma_f16_ss(tmem + kColD, desc_at(dBm, koff_mn(kk)), desc_at(dXwl, koff_mn(kk)), kIdD, 1u);
          ptx::mma_f16_ss(tmem + kColD, desc_at(dBml, koff_mn(kk)), desc_at(dXw, koff_mn(kk)), kIdD, 1u);
        }
      }
      if constexpr (!SO) {
        const Desc dBk = make_desc(opBt, 16u), dCk = make_desc(opCt, 16u);
#pragma unroll
        for (int kk = 0; kk < NS / 16; ++kk) {
          ptx::mma_f16_ss(tmem + kColS, desc_at(dCk, koff_k(kk, 64)), desc_at(dBk, koff_k(kk, 64)),
                           kIdS, kk > 0);
          if constexpr (F32) {
            const Desc dBkl = make_desc(opBt + K::kBtLo, 16u), dCkl = make_desc(opCt + K::kBtLo, 16u);
            ptx::mma_f16_ss(tmem + kColS, desc_at(dCk, koff_k(kk, 64)), desc_at(dBkl, koff_k(kk, 64)),
                             kIdS, 1u);
            ptx::mma_f16_ss(tmem + kColS, desc_at(dCkl, koff_k(kk, 64)), desc_at(dBk, koff_k(kk, 64)),
                             kIdS, 1u);
          }
        }
      }
      ptx::mma_commit(&bar_ds);
      last_commit = &bar_ds;
      last_parity = (uint32_t)(g & 1);
      if constexpr (!SO) {
        if (yoff_ready) {
          const Desc dCk = make_desc(opCt, 16u), dH = make_desc(sbase + K::kH, (uint32_t)NS * 128u);
#pragma unroll
          for (int kk = 0; kk < NS / 16; ++kk) {
            ptx::mma_f16_ss(tmem + kColYo, desc_at(dCk, koff_k(kk, 64)), desc_at(dH, koff_mn(kk)),
                             kIdYo, kk > 0);
            if constexpr (F32) {
              const Desc dCkl = make_desc(opCt + K::kBtLo, 16u);
              const Desc dHl = make_desc(sbase + K::kH + K::kHLo, (uint32_t)NS * 128u);
              ptx::mma_f16_ss(tmem + kColYo, desc_at(dCk, koff_k(kk, 64)), desc_at(dHl, koff_mn(kk)),
                               kIdYo, 1u);
              ptx::mma_f16_ss(tmem + kColYo, desc_at(dCkl, koff_k(kk, 64)), desc_at(dH, koff_mn(kk)),
                               kIdYo, 1u);
            }
          }
        }
        ptx::mma_commit(&bar_yo);
        last_commit = &bar_yo;
      }
    }
    has_state = true;
    if (has_next) {
      load_theta<KP, TPG>(p, nxt, Q, tg, k0, th);
      if (!SO && warp == kDecayWarp) load_decay_raw(p, nxt, Q, lane, dr);
    }

    if constexpr (!SO) {
      // ================================================= mask: P = S o Mask
      wait_or_abort(&bar_ds, (uint32_t)(g & 1), &abort_flag, p.status);
      ptx::tc_fence_after_sync();
      // the bound of the state after D (for its fp16 copy below), published
      // before the mask barrier so that the state phase needs no barrier of
      // its own
      state_ld(hv);
      {
        const float m = warp_max(abs_max(hv));
        if (lane == 0) s_red[warp] = m;
      }
      if (warp == kDecayWarp && has_next) decay_scan(dr, Q, lane, ss[(g + 1) & 1]);
      {
        // thread -> row a, 16 consecutive columns c0 .. c0 + 15 of this warp's half
        const int a = 16 * quad + (lane & 15);
        const int t = a / R;
        const int c0 = 32 * half + 16 * (lane >> 4);
        uint32_t ph_[8], pl_[F32 ? 8 : 1];
        // a warp whose 16 rows x 32 columns lie wholly above the diagonal
        // only writes zeros; elsewhere the mask itself zeroes s > t
        if ((32 * half) / R > (16 * quad + 15) / R) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            ph_[j] = 0u;
            if constexpr (F32) pl_[j] = 0u;
          }
        } else {
          uint32_t sv[16];
          ptx::tmem_ld16_16x32bx2<16>(tmem + kColS + tq + 32u * half, sv);
          ptx::tmem_ld_wait(sv);
          {
            // S -> P units (a power of two: invB invC, times P's scale in F32)
            const float invBC = sc.pmul;
            const float einv = (float)((int)((__float_as_uint(invBC) >> 23) & 0xffu) - 127);
            const float lt = sc.lam2[t] + einv;
            const float gdiag = sc.gam[t] * invBC;
            const int s0 = c0 / R;
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
              // two columns at a time (packed fp32 pairs; same roundings as
              // scalar), their decay terms read as they are needed
              const int u0 = j / R, u1 = (j + 1) / R;
              float2 lsp, wpp;
              if constexpr (R == 1) {
                lsp = *reinterpret_cast<const float2*>(&sc.lam2[s0 + u0]);
                wpp = *reinterpret_cast<const float2*>(&sc.wp[s0 + u0]);
              } else {
                lsp = make_float2(sc.lam2[s0 + u0], sc.lam2[s0 + u1]);
                wpp = make_float2(sc.wp[s0 + u0], sc.wp[s0 + u1]);
              }
              const float2 dl = ptx::sub2(make_float2(lt, lt), lsp);
              const float2 mo = mul2(make_float2(ex2(dl.x), ex2(dl.y)), wpp);
              const float m0 = (s0 + u0 < t) ? mo.x : ((s0 + u0 == t) ? gdiag : 0.f);
              const float m1 = (s0 + u1 < t) ? mo.y : ((s0 + u1 == t) ? gdiag : 0.f);
              const float2 v2 = mul2(make_float2(m0, m1),
                                     make_float2(__uint_as_float(sv[j]), __uint_as_float(sv[j + 1])));
              // fp16 (P is in units of its own scale); F32: and the residual
              const uint32_t hw = pack_f16(v2.x, v2.y);
              ph_[j >> 1] = hw;
              if constexpr (F32) pl_[j >> 1] = f16_residual(hw, v2.x, v2.y);
            }
          }
        }
        const uint32_t o0 = sw128((uint32_t)a, (uint32_t)c0);
        const uint32_t o1 = sw128((uint32_t)a, (uint32_t)c0 + 8u);
        sts128(sbase + K::kPh + o0, make_uint4(ph_[0], ph_[1], ph_[2], ph_[3]));
        sts128(sbase + K::kPh + o1, make_uint4(ph_[4], ph_[5], ph_[6], ph_[7]));
        if constexpr (F32) {
          sts128(sbase + K::kPl + o0, make_uint4(pl_[0], pl_[1], pl_[2], pl_[3]));
          sts128(sbase + K::kPl + o1, make_uint4(pl_[4], pl_[5], pl_[6], pl_[7]));
        }
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before_sync();
      __syncthreads();  // ------------------------------------------ mask
      if (*reinterpret_cast<volatile int*>(&abort_flag)) break;
      if (tid == kMmaTid) {
        // Y = P X
        ptx::tc_fence_after_sync();
        const Desc dPh = make_desc(sbase + K::kPh, 16u);
        const Desc dX = make_desc(sbase + K::kXo, 64u * 128u);
#pragma unroll
        for (int kk = 0; kk < kQR / 16; ++kk)
          ptx::mma_f16_ss(tmem + kColY, desc_at(dPh, koff_k(kk, 64)), desc_at(dX, koff_mn(kk)),
                           kIdY, kk > 0);
        if constexpr (F32) {
          // ... + P_lo X_hi + P_hi X_lo (both tiles are split)
          const Desc dPl = make_desc(sbase + K::kPl, 16u);
          const Desc dXl = make_desc(sbase + K::kXo + K::kXLo, 64u * 128u);
#pragma unroll
          for (int kk = 0; kk < kQR / 16; ++kk)
            ptx::mma_f16_ss(tmem + kColY, desc_at(dPl, koff_k(kk, 64)), desc_at(dX, koff_mn(kk)),
                             kIdY, 1u);
#pragma unroll
          for (int kk = 0; kk < kQR / 16; ++kk)
            ptx::mma_f16_ss(tmem + kColY, desc_at(dPh, koff_k(kk, 64)), desc_at(dXl, koff_mn(kk)),
                             kIdY, 1u);
        }
        ptx::mma_commit(&bar_y);
        last_commit = &bar_y;
      }

      // ================================================= state: fp16 copy
      // (the bound was published before the mask barrier)
      const float uBX = invB * invX;  // the TMEM state is sigma_B sigma_X h
      float h_inv = h_inv_prev;
      if (!last) {
        ptx::tc_fence_after_sync();
        state_ld(hv);
        float m = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) m = fmaxf(m, s_red[w]);
        float h_sig;
        pow2_scale(m * uBX, &h_sig, &h_inv);
        // this chunk's Yoff read the previous copy
        wait_or_abort(&bar_yo, (uint32_t)(g & 1), &abort_flag, p.status);
        write_hcopy(hv, uBX * h_sig);
        ptx::fence_proxy_async_smem();
      }

      // ================================================= output: y = Y + exp(Lam_t) Yoff
      wait_or_abort(&bar_y, (uint32_t)(g & 1), &abort_flag, p.status);
      ptx::tc_fence_after_sync();
      {
        const int a = 16 * quad + (lane & 15);
        const int c0 = 32 * half + 16 * (lane >> 4);  // first p of this thread
        const float el = sc.eL[a / R] * (sc.invC * h_inv_prev);
        uint32_t yv[16];
        ptx::tmem_ld16_16x32bx2<16>(tmem + kColY + tq + 32u * half, yv);
        ptx::tmem_ld_wait(yv);
        float y[16];
        const float ykY = sc.ykY;
#pragma unroll
        for (int j = 0; j < 16; ++j) y[j] = ykY * __uint_as_float(yv[j]);
        if (yoff_ready) {
          uint32_t yo[16];
          ptx::tmem_ld16_16x32bx2<16>(tmem + kColYo + tq + 32u * half, yo);
          ptx::tmem_ld_wait(yo);
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            const float2 r2 = fma2(make_float2(el, el),
                                   make_float2(__uint_as_float(yo[j]), __uint_as_float(yo[j + 1])),
                                   make_float2(y[j], y[j + 1]));
            y[j] = r2.x;
            y[j + 1] = r2.y;
          }
        }
        if constexpr (R == 1) {
          const int64_t t = (int64_t)c * Q + a;
          if (t < p.L) {
            const int64_t e0 = (((int64_t)b * p.L + t) * p.H + h) * kP + c0;
            if constexpr (F32) {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + e0);
#pragma unroll
              for (int q = 0; q < 4; ++q)
                dst[q] = make_float4(y[4 * q], y[4 * q + 1], y[4 * q + 2], y[4 * q + 3]);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + e0);
              dst[0] = make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]),
                                  pack_bf16(y[6], y[7]));
              dst[1] = make_uint4(pack_bf16(y[8], y[9]), pack_bf16(y[10], y[11]),
                                  pack_bf16(y[12], y[13]), pack_bf16(y[14], y[15]));
            }
          }
        } else {
          // staging in the global layout of one chunk: [token][p][r]; bf16 as
          // 128-byte rows of 64 (p, r) elements, 128-byte swizzled like the
          // store's tensor map (without the swizzle a warp's stores hit one
          // bank pair eight times over)
          const int t = a / R, r = a % R;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if constexpr (F32) {
              const uint32_t e = (uint32_t)((t * kP + c0 + j) * R + r);
              asm volatile("st.shared.f32 [%0], %1;" ::"r"(sbase + K::kYs + e * 4u), "f"(y[j])
                           : "memory");
            } else {
              constexpr int kPpr = 64 / R;  // p per 128-byte row
              const int pp = c0 + j;
              const uint32_t row = (uint32_t)(t * R + pp / kPpr);
              const uint32_t inner = (uint32_t)((pp % kPpr) * R + r);
              const uint32_t off = row * 128u + ((((inner >> 3) ^ row) & 7u) << 4) + (inner & 7u) * 2u;
              __nv_bfloat16 v = __float2bfloat16_rn(y[j]);
              sts16(sbase + K::kYs + off, *reinterpret_cast<uint16_t*>(&v));
            }
          }
          ptx::fence_proxy_async_smem();
        }
      }
      h_inv_prev = h_inv;
      yoff_ready = !last;
    } else {
      dsum += sc.lamend2;
    }

    if (last) {
      if constexpr (SO) {
        // the unit's local end state and its (log2 decay, angle) totals
        wait_or_abort(&bar_ds, (uint32_t)(g & 1), &abort_flag, p.status);
        ptx::tc_fence_after_sync();
        state_ld(hv);
        const float uBX = invB * invX;
        float* dst = p.ws_state + sch.unit * (int64_t)NS * kP;
#pragma unroll
        for (int blk = 0; blk < HR / 16; ++blk) {
          uint32_t n, cb;
          hpos(blk, n, cb);
          float4* q4 = reinterpret_cast<float4*>(dst + (int64_t)n * kP + cb);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            q4[j] = make_float4(uBX * hv[16 * blk + 4 * j], uBX * hv[16 * blk + 4 * j + 1],
                                uBX * hv[16 * blk + 4 * j + 2], uBX * hv[16 * blk + 4 * j + 3]);
        }
        float* sd = p.ws_scal + sch.unit * (int64_t)(1 + KP);
        if (tid == 0) sd[0] = dsum;
        if (tid < KP) sd[1 + tid] = s_fang[tid];
      } else if (c == nC - 1 && p.final_state) {
        // final state of the sequence, explicit frame: h = Rot(Phi_{L-1}) g
        // (read from TMEM again rather than kept live through the output phase)
        state_ld(hv);
        const float uBX = invB * invX;
        float* fs = p.final_state + ((int64_t)b * p.heads + h) * NS * kP;
#pragma unroll
        for (int blk = 0; blk < HR / 16; ++blk) {
          uint32_t n, cb;
          hpos(blk, n, cb);
          // the carried angle is wrapped to [-pi, pi]: the fast sincos is accurate there
          float sn, cs;
          __sincosf(s_fang[n >> 1], &sn, &cs);
          const bool odd = n & 1;
          float o[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float hvj = uBX * hv[16 * blk + j];
            const float other = __shfl_xor_sync(0xffffffffu, hvj, 1);
            // even row: c g0 - s g1 ; odd row: s g0 + c g1
            o[j] = odd ? fmaf(sn, other, cs * hvj) : fmaf(-sn, other, cs * hvj);
          }
          float4* dst = reinterpret_cast<float4*>(fs + (int64_t)n * kP + cb);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            dst[j] = make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
        }
      }
    }
    ptx::tc_fence_before_sync();
    // End of the chunk. The full pass at R = 1 needs no barrier here: every
    // shared tile the next chunk overwrites was last read by this chunk's
    // MMAs, whose completion each thread has waited for itself, and the next
    // chunk's first barrier comes before any of its MMAs or TMEM reuse. The
    // state-only pass (decay scan at the end) and R > 1 (the output staging
    // lies over w X, and its TMA store reads it) meet here.
    if constexpr (SO || R > 1) {
      if constexpr (SO) {
        if (warp == kDecayWarp && has_next) decay_scan(dr, Q, lane, ss[(g + 1) & 1]);
      }
      __syncthreads();  // ------------------------------------------ end of chunk
      if (!SO && R > 1 && tid == 0) {
        if constexpr (F32)
          ptx::tma_store_4d(&tm_y, smem + K::kYs, 0, h, c * Q, b);
        else
          ptx::tma_store_5d(&tm_y, smem + K::kYs, 0, 0, h, c * Q, b);
        ptx::tma_store_commit();
      }
      if (*reinterpret_cast<volatile int*>(&abort_flag)) break;
    }
    if (!has_next) break;
    sch = nxt;
  }

  // ---------------------------------------------------------------- teardown
  if (tid == 0) {
    // after an early exit, let issued copies and MMAs finish before the CTA
    // ends (bounded waits): a load still in flight would land in shared
    // memory the CTA no longer owns. After a normal exit these phases are
    // complete already.
    if (raw_pending >= 0) ptx::mbar_wait(&bar_raw, (uint32_t)raw_pending, kWaitNs);
    if (!SO && R > 1) ptx::tma_store_wait_all<0>();
  }
  if (tid == kMmaTid && last_commit) ptx::mbar_wait(last_commit, last_parity, kWaitNs);
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

bool encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* ptr, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return enc(m, dt, (cuuint32_t)rank, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// x / out as a 4-D tensor {P*R, H, L, b}; the box is one head's chunk
// (bf16 with R = 1: 128-byte swizzled, the layout of the X operand).
bool make_act_map(CUtensorMap* m, const void* ptr, const ScanArgs& a) {
  const uint64_t PR = (uint64_t)a.P * a.R, es = a.f32 ? 4 : 2;
  cuuint64_t dims[4] = {PR, (cuuint64_t)a.H, (cuuint64_t)a.L, (cuuint64_t)a.batch};
  cuuint64_t strides[3] = {PR * es, PR * es * a.H, PR * es * a.H * a.L};
  cuuint32_t box[4] = {(cuuint32_t)PR, 1, (cuuint32_t)a.Q, 1};
  return encode(m, a.f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                ptr, dims, strides, box,
                (a.R == 1 && !a.f32) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

// y (the TMA store of R > 1) or x (the load of R = 4) [b, L, H, P, R], bf16:
// a 5-D tensor {64, P*R/64, H, L, b} whose box is one head's chunk as
// 128-byte rows of 64 (p, r) elements, 128-byte swizzled; fp32 keeps the 4-D
// map above.
bool make_out_map(CUtensorMap* m, const void* ptr, const ScanArgs& a) {
  if (a.f32) return make_act_map(m, ptr, a);
  const uint64_t PR = (uint64_t)a.P * a.R;
  cuuint64_t dims[5] = {64, PR / 64, (cuuint64_t)a.H, (cuuint64_t)a.L, (cuuint64_t)a.batch};
  cuuint64_t strides[4] = {128, PR * 2, PR * 2 * a.H, PR * 2 * a.H * a.L};
  cuuint32_t box[5] = {64, (cuuint32_t)(PR / 64), 1, (cuuint32_t)a.Q, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, ptr, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_128B);
}

// B / C [b, L, G, N, R] as a 5-D tensor {d0, N*R/d0, G, L, b} with d0 <= 256.
bool make_bc_map(CUtensorMap* m, const void* ptr, const ScanArgs& a) {
  const uint64_t NR = (uint64_t)a.N * a.R, es = a.f32 ? 4 : 2;
  if (a.R == 4 && !a.f32) {
    // R = 4, bf16: 128-byte rows {64, N R / 64, G, L, b}, 128-byte swizzled
    cuuint64_t dims[5] = {64, NR / 64, (cuuint64_t)a.G, (cuuint64_t)a.L, (cuuint64_t)a.batch};
    cuuint64_t strides[4] = {128, NR * 2, NR * 2 * a.G, NR * 2 * a.G * a.L};
    cuuint32_t box[5] = {64, (cuuint32_t)(NR / 64), 1, (cuuint32_t)a.Q, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, ptr, dims, strides, box,
                  CU_TENSOR_MAP_SWIZZLE_128B);
  }
  const uint64_t d0 = NR < 256 ? NR : 256, d1 = NR / d0;
  cuuint64_t dims[5] = {d0, d1, (cuuint64_t)a.G, (cuuint64_t)a.L, (cuuint64_t)a.batch};
  cuuint64_t strides[4] = {d0 * es, NR * es, NR * es * a.G, NR * es * a.G * a.L};
  cuuint32_t box[5] = {(cuuint32_t)d0, (cuuint32_t)d1, 1, (cuuint32_t)a.Q, 1};
  return encode(m, a.f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5,
                ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// Segmented scan, combine step: for every (sequence, state pair, column),
// walk the segments in order; the state entering segment j+1 is
//   h_{j+1} = Rot(Phi_j) (2^{d_j} h_j + G_j)
// with G_j, d_j, Phi_j the state-only pass's local end state, log2 decay and
// angle of segment j. Entering states overwrite the G's in place.
// The segments' loads are independent of the recurrence, so a thread issues
// them kSegBatch at a time before walking those steps (the walk itself is a
// few flops per segment); the segment angles are wrapped to [-pi, pi], where
// the fast sincos is accurate.
constexpr int kSegBatch = 8;
__global__ void __launch_bounds__(256)
    seg_combine_kernel(float* __restrict__ ws, const float* __restrict__ scal,
                       const float* __restrict__ h_init, int64_t nseq, int nseg, int N, int P) {
  const int KP = N / 2;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= nseq * KP * P) return;
  const int64_t seq = i / ((int64_t)KP * P);
  const int k = (int)((i / P) % KP), pcol = (int)(i % P);
  const int64_t o0 = (int64_t)(2 * k) * P + pcol, o1 = o0 + P;
  // the state entering segment 0: the caller's entering state, or zero
  float h0 = 0.f, h1 = 0.f;
  if (h_init) {
    h0 = h_init[seq * (int64_t)N * P + o0];
    h1 = h_init[seq * (int64_t)N * P + o1];
  }
  for (int j0 = 0; j0 < nseg; j0 += kSegBatch) {
    float g0[kSegBatch], g1[kSegBatch], lg[kSegBatch], ang[kSegBatch];
#pragma unroll
    for (int jj = 0; jj < kSegBatch; ++jj) {
      const int j = j0 + jj;
      if (j < nseg) {
        const int64_t u = seq * nseg + j;
        const float* st = ws + u * (int64_t)N * P;
        const float* sc = scal + u * (int64_t)(1 + KP);
        g0[jj] = st[o0];
        g1[jj] = st[o1];
        lg[jj] = sc[0];
        ang[jj] = sc[1 + k];
      }
    }
#pragma unroll
    for (int jj = 0; jj < kSegBatch; ++jj) {
      const int j = j0 + jj;
      if (j < nseg) {
        float* st = ws + (seq * nseg + j) * (int64_t)N * P;
        st[o0] = h0;  // the state entering segment j
        st[o1] = h1;
        const float d = exp2f(lg[jj]);
        float sn, cs;
        __sincosf(ang[jj], &sn, &cs);
        const float t0 = fmaf(d, h0, g0[jj]), t1 = fmaf(d, h1, g1[jj]);
        h0 = cs * t0 - sn * t1;
        h1 = sn * t0 + cs * t1;
      }
    }
  }
}

struct SegPlan {
  int nseg, seg_chunks;
};

// Whole sequences per work unit, unless there are fewer sequences than SMs:
// then each is cut into segments so that there are about eight units per SM
// (each of at least four chunks).
SegPlan plan_segments(const ScanArgs& a, int sms) {
  const int64_t nseq = a.batch * a.H;
  const int nC = (int)((a.L + a.Q - 1) / a.Q);
  if (nseq >= sms || nC < 8) return {1, nC};
  int64_t target = (8LL * sms + nseq - 1) / nseq;
  if (target > nC / 4) target = nC / 4;
  if (target < 2) return {1, nC};
  const int sc = (int)((nC + target - 1) / target);
  return {(nC + sc - 1) / sc, sc};
}

size_t seg_ws_bytes(const ScanArgs& a, const SegPlan& pl) {
  if (pl.nseg <= 1) return 0;
  const int64_t units = a.batch * a.H * pl.nseg;
  return (size_t)units * (size_t)(a.N * a.P + 1 + a.N / 2) * sizeof(float);
}

int device_sms() {
  const int n = num_sms();
  return n > 0 ? n : 148;
}

template <int R, int NS, bool SO, bool NORM, bool F32>
cudaError_t launch_pass(const CUtensorMap* maps, const TcParams& p, int64_t units, cudaStream_t s) {
  constexpr uint32_t smem = Cfg<R, NS, F32>::kSmem;
  auto kern = scan_tc_kernel<R, NS, SO, NORM, F32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // as much shared memory as the SM has, so that two CTAs fit
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  const int sms = num_sms();
  if (sms <= 0) return cudaErrorInvalidValue;
  // CTAs per SM from the device's limits (shared memory with its per-CTA
  // reservation, registers); each CTA holds 256 of the SM's 512 TMEM
  // columns, so never more than two. Any count is correct: CTAs do not wait
  // on one another.
  int dev = 0, smem_sm = 0, smem_rsv = 0, regs_sm = 0;
  cudaFuncAttributes fa;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
          cudaSuccess ||
      (e = cudaDeviceGetAttribute(&smem_rsv, cudaDevAttrReservedSharedMemoryPerBlock, dev)) !=
          cudaSuccess ||
      (e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev)) !=
          cudaSuccess ||
      (e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess)
    return e;
  const int64_t per_cta_smem = (int64_t)smem + (int64_t)fa.sharedSizeBytes + smem_rsv;
  const int64_t per_cta_regs = (int64_t)((fa.numRegs + 7) / 8 * 8) * kThreads;
  int64_t per_sm = per_cta_smem > 0 ? smem_sm / per_cta_smem : 1;
  if (per_cta_regs > 0 && regs_sm / per_cta_regs < per_sm) per_sm = regs_sm / per_cta_regs;
  per_sm = per_sm < 1 ? 1 : (per_sm > 2 ? 2 : per_sm);
  const int64_t slots = (int64_t)per_sm * sms;
  const unsigned grid = (unsigned)(units < slots ? units : slots);
  kern<<<grid, kThreads, smem, s>>>(maps[0], maps[1], maps[2], maps[3], p);
  return cudaGetLastError();
}

template <int R, int NS, bool NORM, bool F32>
cudaError_t launch_rn(const ScanArgs& a, unsigned int* status, cudaStream_t s) {
  // B, C, x and (R > 1: the output is stored by TMA) y
  CUtensorMap maps[4];
  if (!make_bc_map(&maps[0], a.B, a) || !make_bc_map(&maps[1], a.C, a) ||
      !(R == 4 && !F32 ? make_out_map(&maps[2], a.x, a) : make_act_map(&maps[2], a.x, a)) ||
      !(R > 1 ? make_out_map(&maps[3], a.out, a) : make_act_map(&maps[3], a.x, a)))
    return cudaErrorInvalidValue;
  TcParams p;
  p.dt = a.dt; p.A = a.A; p.lam = a.lam; p.theta = a.theta;
  p.out = a.out;
  p.B_bias = a.B_bias; p.C_bias = a.C_bias;
  p.final_state = a.final_state; p.status = status;
  p.L = a.L; p.H = a.H; p.G = a.G; p.batch = a.batch;
  p.nchunks = (int)((a.L + a.Q - 1) / a.Q);
  p.ws_state = nullptr; p.ws_scal = nullptr;
  p.ws_hin = a.h_init;  // unsegmented: unit u is sequence u
  const SegPlan pl = plan_segments(a, device_sms());
  p.nseg = pl.nseg;
  p.seg_chunks = pl.seg_chunks;
  const int64_t nseq = a.batch * a.H;
  // the kernel indexes units with 32-bit integers (unreachable in practice:
  // 2^31 sequences of x alone would exceed device memory)
  if (nseq * pl.nseg > (int64_t)INT32_MAX) return cudaErrorInvalidValue;
  p.nunits = (int)(nseq * pl.nseg);
  p.heads = (int)a.H;
  p.hpg = (int)(a.H / a.G);
  if (pl.nseg <= 1) return launch_pass<R, NS, false, NORM, F32>(maps, p, nseq, s);
  // segmented: state-only pass, combine, full pass from the entering states
  const size_t need = seg_ws_bytes(a, pl);
  float* ws = static_cast<float*>(a.workspace);
  bool owned = false;
  if (ws == nullptr) {
    cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&ws), need, s);
    if (e != cudaSuccess) return e;
    owned = true;
  } else if (a.workspace_bytes < need) {
    return cudaErrorInvalidValue;
  }
  const int64_t units = nseq * pl.nseg;
  p.ws_state = ws;
  p.ws_scal = ws + units * a.N * a.P;
  p.final_state = nullptr;
  p.ws_hin = nullptr;  // the state-only pass starts every segment from zero
  cudaError_t e = launch_pass<R, NS, true, NORM, F32>(maps, p, units, s);
  if (e == cudaSuccess) {
    const int64_t n = nseq * (a.N / 2) * a.P;
    seg_combine_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(ws, p.ws_scal, a.h_init, nseq,
                                                                   pl.nseg, (int)a.N, (int)a.P);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    p.ws_state = nullptr;
    p.ws_hin = ws;
    p.final_state = a.final_state;
    e = launch_pass<R, NS, false, NORM, F32>(maps, p, units, s);
  }
  if (owned) {
    const cudaError_t f = cudaFreeAsync(ws, s);
    if (e == cudaSuccess) e = f;
  }
  return e;
}

}  // namespace

size_t scan_tc_workspace_bytes(const ScanArgs& a) {
  if (!scan_tc_supported(a.N, a.P, a.R, a.Q)) return 0;
  return seg_ws_bytes(a, plan_segments(a, device_sms()));
}

bool scan_tc_supported(int64_t N, int64_t P, int R, int Q) {
  if (P != kP) return false;
  if (N != 64 && N != 128) return false;
  if (!(R == 1 || R == 2 || R == 4)) return false;
  return Q * R == kQR;
}

cudaError_t launch_scan_tc(const ScanArgs& a, unsigned int* status, cudaStream_t s) {
  if (a.L > 0x7fffffffLL - 2 * kQR || a.batch > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int key = a.R * 1000 + (int)a.N;
  if (a.bc_norm && a.f32) return cudaErrorInvalidValue;  // BCNorm is fused on the bf16 path only
  if (a.bc_norm) {
    switch (key) {
      case 1064: return launch_rn<1, 64, true, false>(a, status, s);
      case 1128: return launch_rn<1, 128, true, false>(a, status, s);
      case 2064: return launch_rn<2, 64, true, false>(a, status, s);
      case 2128: return launch_rn<2, 128, true, false>(a, status, s);
      case 4064: return launch_rn<4, 64, true, false>(a, status, s);
      case 4128: return launch_rn<4, 128, true, false>(a, status, s);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (key) {
    case 1064: return a.f32 ? launch_rn<1, 64, false, true>(a, status, s)
                      : launch_rn<1, 64, false, false>(a, status, s);
    case 1128: return a.f32 ? launch_rn<1, 128, false, true>(a, status, s)
                      : launch_rn<1, 128, false, false>(a, status, s);
    case 2064: return a.f32 ? launch_rn<2, 64, false, true>(a, status, s)
                      : launch_rn<2, 64, false, false>(a, status, s);
    case 2128: return a.f32 ? launch_rn<2, 128, false, true>(a, status, s)
                      : launch_rn<2, 128, false, false>(a, status, s);
    case 4064: return a.f32 ? launch_rn<4, 64, false, true>(a, status, s)
                      : launch_rn<4, 64, false, false>(a, status, s);
    case 4128: return a.f32 ? launch_rn<4, 128, false, true>(a, status, s)
                      : launch_rn<4, 128, false, false>(a, status, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace m3
