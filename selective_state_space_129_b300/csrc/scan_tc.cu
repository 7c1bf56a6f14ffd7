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
// each scaled by a power of two chosen per chunk from a bound of its
// magnitude, so fp16's range never limits the inputs. The scales are undone
// exactly where a per-element factor is applied anyway (mask, state update,
// output). P is split into bf16 high and low parts so that P X (X is an exact
// bf16 input) keeps ~16 significant bits. The cumulative angle is carried
// from chunk to chunk as a float-float pair fed by Kahan-compensated sums, so
// it does not drift over long sequences.
//
// Organisation: a persistent, warp-specialised CTA (512 threads, one per SM)
// walks work units (whole (b, h) sequences, or segments of them when there
// are fewer sequences than SMs), chunk by chunk, as a software pipeline:
//   warps 0-7    prologue: decay scan (warp 0), angles, RoPE fold of B/C into
//                fp16 UMMA tiles, w X, into one of two operand slots per chunk;
//                one thread issues the TMA of the next chunk's raw B, C,
//                theta, x tiles (one raw slot), two others the chunk's S and D
//                MMAs into one of two TMEM accumulator sets; one warp
//                prefetches the next chunk's dt, lambda
//   warps 8-15   core (two warps per TMEM lane quadrant, 32 columns each):
//                mask S -> P, state H = exp(Lam_end) H + D and its fp16 copy,
//                y = Y + exp(Lam_t) Yoff -> TMA store, final state; its thread
//                0 issues Y = P X for chunk c and Yoff = Ct H for chunk c+1,
//                overlapping chunk c's epilogue
// so the prologue of chunk c+1 runs while the core finishes chunk c. Roles
// hand off through mbarriers; a role synchronises internally with its own
// named barrier. Operand tiles are 128-byte-swizzled rows of 64 16-bit
// elements; a [rows][64k] tile is at once the K-major operand along its
// columns and the MN-major operand along its rows, so Bt serves both S (K = N)
// and the state GEMM (K = tokens).
// Every mbarrier wait is bounded; on expiry the CTA records the status word,
// every role leaves its loop at the next chunk boundary, and the CTA still
// frees its tensor memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace m3 {
namespace {

constexpr int kProWarps = 8, kCoreWarps = 8;
constexpr int kProThreads = kProWarps * 32;    // 256
constexpr int kCoreThreads = kCoreWarps * 32;  // 256: two warps per TMEM lane quadrant
constexpr int kThreads = kProThreads + kCoreThreads;  // 512 (128 registers per thread)
constexpr int kWarpTmem = kProWarps;                  // allocates / frees TMEM
constexpr uint32_t kBarPro = 1, kBarCore = 2;          // named barrier ids
constexpr int kQR = 64;  // rows of the flattened (token, rank) tile
constexpr int kP = 64;   // head dim of the tensor-core path
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemSlot = 256;          // columns per accumulator set
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

// TMEM column offsets of the four fp32 accumulators within a set.
constexpr uint32_t kColS = 0, kColD = 64, kColY = 128, kColYo = 192;

constexpr uint32_t align1k(uint32_t v) { return (v + 1023u) & ~1023u; }

template <int R, int NS>
struct Cfg {
  static constexpr int Q = kQR / R;          // tokens per chunk
  static constexpr int KP = NS / 2;          // rotating state pairs
  static constexpr int KP2 = KP / 2;         // pair-pairs: a prologue thread owns two pairs
  static constexpr int TG = kProThreads / KP2;  // token groups in the prologue
  static constexpr int TPG = Q / TG;         // tokens per prologue thread
  static_assert(TPG >= 1 && Q % TG == 0, "token groups must divide the chunk");
  static constexpr int HR = NS * kP / kCoreThreads;  // fp32 state values per core thread
  static constexpr int BW = 2 * R;           // raw 32-bit words of B (or C) per token and thread
  // raw slot (TMA destination): B, C [Q][NS*R] bf16, theta [Q][KP] fp32, x [Q][P*R] bf16
  static constexpr uint32_t kRawB = 0;
  static constexpr uint32_t kRawC = kRawB + Q * NS * R * 2;
  static constexpr uint32_t kRawTh = kRawC + Q * NS * R * 2;
  static constexpr uint32_t kRawX = align1k(kRawTh + Q * KP * 4);  // 128B-swizzled for R = 1
  static constexpr uint32_t kRawBytes = kRawX + (uint32_t)(Q * kP * R * 2);
  // two operand slots: Bt, Ct [64][NS] fp16, w X [64][64] fp16, X [64][64] bf16
  static constexpr uint32_t kOpBt = 0;
  static constexpr uint32_t kOpCt = 64 * NS * 2;
  static constexpr uint32_t kOpXw = 2 * 64 * NS * 2;
  static constexpr uint32_t kOpXo = kOpXw + kTileBytes;
  static constexpr uint32_t kOpBytes = kOpXo + kTileBytes;
  static constexpr uint32_t kOp0 = align1k(kRawBytes);
  // core tiles: P high / low (bf16), fp16 state copy [NS][64], output staging
  static constexpr uint32_t kPh = kOp0 + 2 * kOpBytes;
  static constexpr uint32_t kPl = kPh + kTileBytes;
  static constexpr uint32_t kH = kPl + kTileBytes;
  static constexpr uint32_t kYs = kH + NS * 128;
  static constexpr uint32_t kBytes = kYs + kTileBytes;
  static constexpr uint32_t kSmem = kBytes + 1024;  // + alignment slack
  // bytes landing on the raw barrier per chunk
  static constexpr uint32_t kTxBytes =
      2u * Q * NS * R * 2 + (uint32_t)(Q * KP * 4) + (uint32_t)(Q * kP * R * 2);
};

// Per-chunk scalars handed from the prologue to the core (one set per slot).
template <int KP>
struct __align__(16) SlotScalars {
  float lam2[64];  // Lam_t in log2 units
  float gam[64];   // gamma_t
  float wp[64];    // gamma_t + bhat_{t+1}
  float eL[64];    // exp(Lam_t)
  float wend[64];  // exp(Lam_end - Lam_t) (gamma_t + bhat_{t+1})
  float fang[KP];  // cumulative angle after the chunk (last chunk of a sequence)
  float eLend, wmax, invB, invC, invX;
  float lamend2;  // Lam_end in log2 units
  float pad[2];
};

struct TcParams {
  const float* dt;
  const float* A;
  const float* lam;
  const float* B_bias;
  const float* C_bias;
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
// element e of a run of bf16 values packed two per word (little-endian)
template <int N>
__device__ __forceinline__ float bf_at(const uint32_t (&w)[N], int e) {
  return (e & 1) ? bf_hi(w[e >> 1]) : bf_lo(w[e >> 1]);
}
// largest magnitude held in an accumulator of bf16x2 abs-maxima, as a float
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

using ptx::add2;
using ptx::fma2;
using ptx::mul2;
using ptx::sub2;

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
// CTA's abort flag. Returns false if the CTA is (now) aborting.
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
// the sequence; a CTA walks units blockIdx.x, +gridDim.x, ... chunk by chunk
// (g counts its chunks; slots and mbarrier phases follow g).
// (32-bit indices, divided once per unit: 64-bit division is a long
// software sequence that would sit on the per-chunk critical path).
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
// lane + 32. Only loads: the arithmetic waits until the values are needed, so
// that the load latency overlaps other work.
struct DecayRaw {
  float dt[2], lam[2], dtn[2], lamn[2];
};
__device__ __forceinline__ void load_decay_raw(const TcParams& p, int64_t b, int64_t h, int64_t t0,
                                               int Q, int lane, DecayRaw& d) {
  const int64_t L = p.L, H = p.H;
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
}
// dt, lambda and bhat of the successor into the chunk's decay-input buffer
__device__ __forceinline__ void store_decay(const DecayRaw& d, int lane, float* sdt, float* slam,
                                            float* sbn) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    sdt[lane + 32 * j] = d.dt[j];
    slam[lane + 32 * j] = d.lam[j];
    sbn[lane + 32 * j] = (1.f - d.lamn[j]) * d.dtn[j];
  }
}

// SO: the state-only pass of a segmented scan (no C, no outputs).
template <int R, int NS, bool SO>
__global__ void __launch_bounds__(kThreads, 1)
    scan_tc_kernel(const __grid_constant__ CUtensorMap tm_B, const __grid_constant__ CUtensorMap tm_C,
                   const __grid_constant__ CUtensorMap tm_th, const __grid_constant__ CUtensorMap tm_x,
                   const __grid_constant__ CUtensorMap tm_y, TcParams p) {
  using K = Cfg<R, NS>;
  constexpr int Q = K::Q, KP = K::KP, KP2 = K::KP2, TG = K::TG, TPG = K::TPG, HR = K::HR;
  constexpr uint32_t kIdS = ptx::idesc_f16_f32(64, 64, false, false);
  constexpr uint32_t kIdD = ptx::idesc_f16_f32(NS, 64, true, true);
  constexpr uint32_t kIdYo = ptx::idesc_f16_f32(64, 64, false, true);
  constexpr uint32_t kIdY = ptx::idesc_bf16_f32(64, 64, false, true);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_addr(smem);

  __shared__ uint64_t bar_raw_full;
  __shared__ uint64_t bar_op_full[2], bar_slot_free[2], bar_acc_full[2], bar_y_full[2];
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_flag;
  __shared__ int s_go[2];  // per-role broadcast of "continue" decisions
  __shared__ SlotScalars<KP> ss[2];
  __shared__ float s_dtraw[2][64], s_lamraw[2][64], s_bnx[2][64];
  __shared__ __align__(16) float s_tot[2][TG][KP];   // per token group: angle total (hi, lo)
  __shared__ float s_carry[2][2][KP];  // [chunk parity][hi, lo][pair]
  __shared__ unsigned int s_max[2][3];  // per chunk parity: bounds of |B|, |C|, |x| (float bits)
  __shared__ float s_hred[kCoreWarps];
  __shared__ float s_bias_red[2][kProWarps];
  // R > 1: the head's B / C bias transposed to [rank][row] (registers for R = 1)
  __shared__ __align__(16) float s_biasT[2][R][NS];  // B, C bias of the head, [rank][n]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nC = p.nchunks;

  // ---------------------------------------------------------------- setup
  if (warp == kWarpTmem) {
    ptx::tmem_alloc(&tmem_holder, kTmemCols);
    ptx::tmem_relinquish();
  }
  if (tid == 0) {
    abort_flag = 0;
    for (int i = 0; i < 6; ++i) (&s_max[0][0])[i] = 0u;
    ptx::mbar_init(&bar_raw_full, 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&bar_op_full[s], 1);
      ptx::mbar_init(&bar_slot_free[s], kCoreWarps);
      ptx::mbar_init(&bar_acc_full[s], SO ? 1 : 2);  // the S and the D issuer commit
      ptx::mbar_init(&bar_y_full[s], 1);
    }
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&tm_B);
    ptx::prefetch_tensormap(&tm_C);
    ptx::prefetch_tensormap(&tm_th);
    ptx::prefetch_tensormap(&tm_x);
    ptx::prefetch_tensormap(&tm_y);
  }
  // masked-score tiles: blocks above the diagonal are zero and never written again
  for (uint32_t i = tid * 16; i < 2u * kTileBytes; i += kThreads * 16)
    sts128(sbase + K::kPh + i, make_uint4(0, 0, 0, 0));
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem = tmem_holder;

  // TMA of one chunk's raw tiles into the raw slot (one prologue thread)
  auto issue_raw = [&](const Sched& u) {
    const int b = u.b, h = u.h, gi = h / p.hpg;
    const int t0 = u.c * Q;
    ptx::mbar_arrive_expect_tx(&bar_raw_full, SO ? K::kTxBytes - K::kRawC : K::kTxBytes);
    ptx::tma_load_5d(smem + K::kRawB, &tm_B, &bar_raw_full, 0, 0, gi, t0, b);
    if (!SO) ptx::tma_load_5d(smem + K::kRawC, &tm_C, &bar_raw_full, 0, 0, gi, t0, b);
    ptx::tma_load_4d(smem + K::kRawTh, &tm_th, &bar_raw_full, 0, gi, t0, b);
    ptx::tma_load_4d(smem + K::kRawX, &tm_x, &bar_raw_full, 0, h, t0, b);
  };

  if (warp < kProWarps) {
    // ============================================================ prologue
    const int kk2 = tid % KP2, tg = tid / KP2;
    const int k0 = 2 * kk2;  // this thread's pairs: k0, k0 + 1 (rows 4kk2 .. 4kk2 + 3)
    int cur_h = -1;
    float bmax_bias = 0.f, cmax_bias = 0.f;
    int inflight = -1;  // phase parity of a raw load issued and not yet consumed
    // the first chunk's inputs
    Sched sch;
    sch.start(blockIdx.x, p);
    // one-off duties sit on warps without other extra work: TMA of the raw
    // tiles (warp 4), S and D MMA issue (warps 2 and 3); warp 0 runs the decay
    // scan, warp 1 loads the next chunk's decay inputs, warps 6 and 7 carry
    // the angle totals
    constexpr int kTmaTid = 128, kSTid = 64, kDTid = 96;
    if (tid == kTmaTid) {
      issue_raw(sch);
      inflight = 0;
    }
    if (warp == 1) {
      DecayRaw d;
      load_decay_raw(p, sch.b, sch.h, (int64_t)sch.c * Q, Q, lane, d);
      store_decay(d, lane, s_dtraw[0], s_lamraw[0], s_bnx[0]);
    }
    // the first chunk's decay inputs are in place before warp 0 reads them
    // (later chunks' are stored before the previous chunk's last barrier)
    ptx::named_bar_sync(kBarPro, kProThreads);
    float A_h = 0.f;
    for (int g = 0;; ++g) {
      const int h = sch.h;
      const int c = sch.c, s = g & 1, db = g & 1;
      const bool has_next = sch.c + 1 < sch.c_end || sch.unit + (int)gridDim.x < p.nunits;
      SlotScalars<KP>& sc = ss[s];
      if (h != cur_h) {
        // per-head A, bias (fp32) and a block-wide bound of the bias magnitude
        cur_h = h;
        A_h = p.A[h];
        float mb = 0.f, mc = 0.f;
        // the previous head's bias was last read before the previous chunk's
        // last barrier
        for (int i = tid; i < NS * R; i += kProThreads) {
          const float vb = p.B_bias ? p.B_bias[(int64_t)h * NS * R + i] : 0.f;
          const float vc = p.C_bias ? p.C_bias[(int64_t)h * NS * R + i] : 0.f;
          s_biasT[0][i % R][i / R] = vb;
          s_biasT[1][i % R][i / R] = vc;
          mb = fmaxf(mb, fabsf(vb));
          mc = fmaxf(mc, fabsf(vc));
        }
        mb = warp_max(mb);
        mc = warp_max(mc);
        if (lane == 0) {
          s_bias_red[0][warp] = mb;
          s_bias_red[1][warp] = mc;
        }
        ptx::named_bar_sync(kBarPro, kProThreads);
        bmax_bias = 0.f;
        cmax_bias = 0.f;
#pragma unroll
        for (int w = 0; w < kProWarps; ++w) {
          bmax_bias = fmaxf(bmax_bias, s_bias_red[0][w]);
          cmax_bias = fmaxf(cmax_bias, s_bias_red[1][w]);
        }
      }
      // 1. every thread waits for this chunk's raw tiles itself (no block
      // barrier here); an expired wait sets the abort flag, which every thread
      // reads after the next barrier
      if (wait_or_abort(&bar_raw_full, (uint32_t)(g & 1), &abort_flag, p.status) && tid == kTmaTid)
        inflight = -1;
      // 2b. raw tiles -> registers (loads issued first)
      float2 th2[TPG];
      uint32_t bw[TPG][K::BW], cw[TPG][K::BW];
      uint32_t bacc = 0u, cacc = 0u;
#pragma unroll
      for (int i = 0; i < TPG; ++i) {
        const int t = tg * TPG + i;
        const uint2 tv = lds64(sbase + K::kRawTh + (uint32_t)(t * KP + k0) * 4u);
        th2[i] = make_float2(__uint_as_float(tv.x), __uint_as_float(tv.y));
        const uint32_t ob = (uint32_t)(t * NS * R + 4 * kk2 * R) * 2u;
        if constexpr (R == 1) {
          const uint2 vb = lds64(sbase + K::kRawB + ob);
          bw[i][0] = vb.x; bw[i][1] = vb.y;
          if constexpr (!SO) {
            const uint2 vc = lds64(sbase + K::kRawC + ob);
            cw[i][0] = vc.x; cw[i][1] = vc.y;
          }
        } else {
#pragma unroll
          for (int q = 0; q < K::BW / 4; ++q) {
            const uint4 vb = lds128(sbase + K::kRawB + ob + 16u * q);
            bw[i][4 * q] = vb.x; bw[i][4 * q + 1] = vb.y; bw[i][4 * q + 2] = vb.z; bw[i][4 * q + 3] = vb.w;
            if constexpr (!SO) {
              const uint4 vc = lds128(sbase + K::kRawC + ob + 16u * q);
              cw[i][4 * q] = vc.x; cw[i][4 * q + 1] = vc.y; cw[i][4 * q + 2] = vc.z; cw[i][4 * q + 3] = vc.w;
            }
          }
        }
      }
      // 2a (while the tile loads above are in flight). Decay scan (warp 0, once
      // operand slot s and its scalars are free:
      // the rest of the slot is written after the next barrier); the next
      // chunk's dt, lambda (warp 1, into registers)
      DecayRaw nd;
      int slot_ok = 1;
      if (warp == 0 && g >= 2) {
        if (lane == 0)
          slot_ok = wait_or_abort(&bar_slot_free[s], (uint32_t)(((g >> 1) & 1) ^ 1), &abort_flag,
                                  p.status) ? 1 : 0;
        slot_ok = __shfl_sync(0xffffffffu, slot_ok, 0);
      }
      if (warp == 0 && slot_ok) {
        float dtv[2], lmv[2], bnx[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int i = lane + 32 * j;
          dtv[j] = s_dtraw[db][i];
          lmv[j] = s_lamraw[db][i];
          bnx[j] = s_bnx[db][i];
        }
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
        const float lv[2] = {a0, a1};
        float wm = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int i = lane + 32 * j;
          if (i < Q) {
            const float gam = lmv[j] * dtv[j];
            const float wpv = gam + bnx[j];
            const float we = ex2(lam_end - lv[j]) * wpv;
            sc.lam2[i] = lv[j];
            sc.gam[i] = gam;
            sc.wp[i] = wpv;
            sc.wend[i] = we;
            sc.eL[i] = ex2(lv[j]);
            wm = fmaxf(wm, fabsf(we));
          }
        }
        wm = warp_max(wm);
        if (lane == 0) {
          sc.eLend = ex2(lam_end);
          sc.lamend2 = lam_end;
          sc.wmax = wm;
        }
      } else if (warp == 1 && has_next) {
        Sched nxt = sch;
        nxt.next(p);
        load_decay_raw(p, nxt.b, nxt.h, (int64_t)nxt.c * Q, Q, lane, nd);
      }
      // 2c. magnitude bounds, Kahan-compensated angle sums
#pragma unroll
      for (int i = 0; i < TPG; ++i) {
#pragma unroll
        for (int q = 0; q < K::BW; ++q) {
          bacc = ptx::bf16x2_absmax(bacc, bw[i][q]);
          if constexpr (!SO) cacc = ptx::bf16x2_absmax(cacc, cw[i][q]);
        }
      }
      float2 ph[TPG];
      {
        float2 run = make_float2(0.f, 0.f), comp = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < TPG; ++i) {
          const float d = s_dtraw[db][tg * TPG + i];
          const float2 yk = sub2(mul2(make_float2(d, d), th2[i]), comp);
          const float2 tk = add2(run, yk);
          comp = sub2(sub2(tk, run), yk);
          run = tk;
          ph[i] = run;
        }
        s_tot[0][tg][k0] = run.x;
        s_tot[0][tg][k0 + 1] = run.y;
        s_tot[1][tg][k0] = -comp.x;
        s_tot[1][tg][k0 + 1] = -comp.y;
      }
      // x of this chunk -> registers (w X and the operand copy of X)
      constexpr int kXItems = (R == 1) ? 2 : (Q * (kP / 4)) / kProThreads;
      constexpr int kXVec = (R == 1) ? 1 : R / 2;
      uint4 xv[kXItems][kXVec];
      uint32_t xacc = 0u;
      const uint32_t opb = sbase + K::kOp0 + (uint32_t)s * K::kOpBytes;
#pragma unroll
      for (int j = 0; j < kXItems; ++j) {
        const int it = tid + kProThreads * j;
        if constexpr (R == 1) {
          xv[j][0] = lds128(sbase + K::kRawX + (uint32_t)it * 16u);  // 16-byte chunk, row it / 8
        } else {
          const int sx = it / (kP / 4), pb = it % (kP / 4);
          const uint32_t src = sbase + K::kRawX + (uint32_t)(sx * kP * R + 4 * pb * R) * 2u;
#pragma unroll
          for (int q = 0; q < kXVec; ++q) xv[j][q] = lds128(src + 16u * q);
        }
#pragma unroll
        for (int q = 0; q < kXVec; ++q) {
          xacc = ptx::bf16x2_absmax(xacc, xv[j][q].x);
          xacc = ptx::bf16x2_absmax(xacc, xv[j][q].y);
          xacc = ptx::bf16x2_absmax(xacc, xv[j][q].z);
          xacc = ptx::bf16x2_absmax(xacc, xv[j][q].w);
        }
      }
      {
        // non-negative floats order like their bit patterns
        const float bm = warp_max(bf_absmax(bacc)), cm = warp_max(bf_absmax(cacc));
        const float xm = warp_max(bf_absmax(xacc));
        if (lane == 0) {
          atomicMax(&s_max[g & 1][0], __float_as_uint(bm));
          atomicMax(&s_max[g & 1][1], __float_as_uint(cm));
          atomicMax(&s_max[g & 1][2], __float_as_uint(xm));
        }
      }
      ptx::named_bar_sync(kBarPro, kProThreads);
      if (*reinterpret_cast<volatile int*>(&abort_flag)) break;  // uniform after the barrier
      // every read of the raw slot is done: refill it with the next chunk
      if (has_next) {
        if (tid == kTmaTid) {
          Sched nxt = sch;
          nxt.next(p);
          issue_raw(nxt);
          inflight = (g + 1) & 1;
        }
        if (warp == 1) store_decay(nd, lane, s_dtraw[db ^ 1], s_lamraw[db ^ 1], s_bnx[db ^ 1]);
      }
      // 3. per-chunk fp16 scales of Bt, Ct and w X
      float sigB, invB, sigC, invC, sigX, invX;
      {
        const float mb = __uint_as_float(s_max[g & 1][0]);
        const float mc = __uint_as_float(s_max[g & 1][1]);
        const float mx = __uint_as_float(s_max[g & 1][2]);
        // the other parity's words are free (read last chunk): clear them for the next
        if (tid == 0) {
          s_max[(g + 1) & 1][0] = 0u;
          s_max[(g + 1) & 1][1] = 0u;
          s_max[(g + 1) & 1][2] = 0u;
        }
        // a rotated pair keeps its norm: |Rot(v)_i| <= sqrt(2) max|v| < 2 max|v|
        pow2_scale(2.f * (mb + bmax_bias), &sigB, &invB);
        pow2_scale(2.f * (mc + cmax_bias), &sigC, &invC);
        pow2_scale(mx * sc.wmax, &sigX, &invX);
        if (tid == 0) {
          sc.invB = invB;
          sc.invC = invC;
          sc.invX = invX;
        }
      }
      // 4. angle before this thread's first token: carry + earlier groups.
      // Within the chunk an fp32 offset suffices; the carry to the next
      // chunk is float-float so that it does not drift.
      const int cpar = g & 1;
      float2 off;
      {
        float o0 = 0.f, o1 = 0.f;
        for (int q = 0; q < tg; ++q) {
          const float2 hi = *reinterpret_cast<const float2*>(&s_tot[0][q][k0]);
          const float2 lo = *reinterpret_cast<const float2*>(&s_tot[1][q][k0]);
          const float2 o = add2(make_float2(o0, o1), add2(hi, lo));
          o0 = o.x;
          o1 = o.y;
        }
        float ch0 = 0.f, cl0 = 0.f, ch1 = 0.f, cl1 = 0.f;
        if (c > sch.c_begin) {
          ch0 = s_carry[cpar][0][k0];
          cl0 = s_carry[cpar][1][k0];
          ch1 = s_carry[cpar][0][k0 + 1];
          cl1 = s_carry[cpar][1][k0 + 1];
        }
        off.x = wrap_rad(ch0 + (cl0 + o0));
        off.y = wrap_rad(ch1 + (cl1 + o1));
        // the carry of pair k0 is updated by group TG-1, that of k0+1 by TG-2
        if (tg >= TG - 2) {
          const int k = (tg == TG - 1) ? k0 : k0 + 1;
          // float-float sum of the group totals as a tree, then the carry
          float th[TG], tl[TG];
#pragma unroll
          for (int q = 0; q < TG; ++q) {
            th[q] = s_tot[0][q][k];
            tl[q] = s_tot[1][q][k];
          }
#pragma unroll
          for (int w = 1; w < TG; w <<= 1)
#pragma unroll
            for (int q = 0; q + w < TG; q += 2 * w) ff_add(th[q], tl[q], th[q + w], tl[q + w]);
          float eh = (tg == TG - 1) ? ch0 : ch1, el = (tg == TG - 1) ? cl0 : cl1;
          ff_add(eh, el, th[0], tl[0]);
          ff_wrap(eh, el);
          s_carry[cpar ^ 1][0][k] = eh;
          s_carry[cpar ^ 1][1][k] = el;
          if (c == sch.c_end - 1) sc.fang[k] = eh + el;
        }
      }
      // 5. RoPE fold: sigma Rot(-Phi) (B + bias), likewise C, into fp16 tiles
      {
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < TPG; ++i) {
          ph[i] = add2(off, ph[i]);
          amax = fmaxf(amax, fmaxf(fabsf(ph[i].x), fabsf(ph[i].y)));
        }
        if (__any_sync(0xffffffffu, amax > kAngleDirect)) {
#pragma unroll
          for (int i = 0; i < TPG; ++i) ph[i] = make_float2(wrap_rad(ph[i].x), wrap_rad(ph[i].y));
        }
      }
      const float2 sB2 = make_float2(sigB, sigB), sC2 = make_float2(sigC, sigC);
      if constexpr (R == 1) {
        // sigma (B + bias) = fma(sigma, B, sigma bias), exact for a power-of-two
        // sigma, so the scale rides on the bias add instead of on cos and sin
        const float4 bq = *reinterpret_cast<const float4*>(&s_biasT[0][0][4 * kk2]);
        const float2 bs0 = mul2(sB2, make_float2(bq.x, bq.z)), bs1 = mul2(sB2, make_float2(bq.y, bq.w));
        float2 cs0 = make_float2(0.f, 0.f), cs1 = cs0;
        if constexpr (!SO) {
          const float4 cq = *reinterpret_cast<const float4*>(&s_biasT[1][0][4 * kk2]);
          cs0 = mul2(sC2, make_float2(cq.x, cq.z));
          cs1 = mul2(sC2, make_float2(cq.y, cq.w));
        }
#pragma unroll
        for (int i = 0; i < TPG; ++i) {
          float2 sn, cs;
          __sincosf(ph[i].x, &sn.x, &cs.x);
          __sincosf(ph[i].y, &sn.y, &cs.y);
          const float2 nsn = make_float2(-sn.x, -sn.y);
          const int t = tg * TPG + i;
          // .x holds pair k0 (rows 4kk2, 4kk2 + 1), .y pair k0 + 1
          const float2 b0 = fma2(sB2, make_float2(bf_at(bw[i], 0), bf_at(bw[i], 2)), bs0);
          const float2 b1 = fma2(sB2, make_float2(bf_at(bw[i], 1), bf_at(bw[i], 3)), bs1);
          // Rot(-Phi) = [[cos, sin], [-sin, cos]]
          const float2 bt0 = fma2(cs, b0, mul2(sn, b1)), bt1 = fma2(cs, b1, mul2(nsn, b0));
          const uint32_t o = tile_off((uint32_t)t, 4u * kk2, 64u);
          sts64(opb + K::kOpBt + o, pack_f16(bt0.x, bt1.x), pack_f16(bt0.y, bt1.y));
          if constexpr (!SO) {
            const float2 c0 = fma2(sC2, make_float2(bf_at(cw[i], 0), bf_at(cw[i], 2)), cs0);
            const float2 c1 = fma2(sC2, make_float2(bf_at(cw[i], 1), bf_at(cw[i], 3)), cs1);
            const float2 ct0 = fma2(cs, c0, mul2(sn, c1)), ct1 = fma2(cs, c1, mul2(nsn, c0));
            sts64(opb + K::kOpCt + o, pack_f16(ct0.x, ct1.x), pack_f16(ct0.y, ct1.y));
          }
        }
      } else if constexpr (TPG <= 2) {
        // few tokens per thread (R = 4): every rank's bias row is loaded once
        // and applied to the thread's tokens, whose cos / sin are kept
        float2 csB[TPG], snB[TPG], nsnB[TPG], csC[TPG], snC[TPG], nsnC[TPG];
#pragma unroll
        for (int i = 0; i < TPG; ++i) {
          float2 sn, cs;
          __sincosf(ph[i].x, &sn.x, &cs.x);
          __sincosf(ph[i].y, &sn.y, &cs.y);
          csB[i] = mul2(cs, sB2);
          snB[i] = mul2(sn, sB2);
          nsnB[i] = make_float2(-snB[i].x, -snB[i].y);
          csC[i] = mul2(cs, sC2);
          snC[i] = mul2(sn, sC2);
          nsnC[i] = make_float2(-snC[i].x, -snC[i].y);
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float4 bq = *reinterpret_cast<const float4*>(&s_biasT[0][r][4 * kk2]);
          float4 cq = bq;
          if constexpr (!SO) cq = *reinterpret_cast<const float4*>(&s_biasT[1][r][4 * kk2]);
#pragma unroll
          for (int i = 0; i < TPG; ++i) {
            const int t = tg * TPG + i;
            float2 b0 = make_float2(bf_at(bw[i], 0 * R + r), bf_at(bw[i], 2 * R + r));
            float2 b1 = make_float2(bf_at(bw[i], 1 * R + r), bf_at(bw[i], 3 * R + r));
            b0 = add2(b0, make_float2(bq.x, bq.z));
            b1 = add2(b1, make_float2(bq.y, bq.w));
            const float2 bt0 = fma2(csB[i], b0, mul2(snB[i], b1));
            const float2 bt1 = fma2(csB[i], b1, mul2(nsnB[i], b0));
            const uint32_t o = tile_off((uint32_t)(t * R + r), 4u * kk2, 64u);
            sts64(opb + K::kOpBt + o, pack_f16(bt0.x, bt1.x), pack_f16(bt0.y, bt1.y));
            if constexpr (!SO) {
              float2 c0 = make_float2(bf_at(cw[i], 0 * R + r), bf_at(cw[i], 2 * R + r));
              float2 c1 = make_float2(bf_at(cw[i], 1 * R + r), bf_at(cw[i], 3 * R + r));
              c0 = add2(c0, make_float2(cq.x, cq.z));
              c1 = add2(c1, make_float2(cq.y, cq.w));
              const float2 ct0 = fma2(csC[i], c0, mul2(snC[i], c1));
              const float2 ct1 = fma2(csC[i], c1, mul2(nsnC[i], c0));
              sts64(opb + K::kOpCt + o, pack_f16(ct0.x, ct1.x), pack_f16(ct0.y, ct1.y));
            }
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < TPG; ++i) {
          float2 sn, cs;
          __sincosf(ph[i].x, &sn.x, &cs.x);
          __sincosf(ph[i].y, &sn.y, &cs.y);
          const float2 csB = mul2(cs, sB2), snB = mul2(sn, sB2);
          const float2 csC = mul2(cs, sC2), snC = mul2(sn, sC2);
          const float2 nsnB = make_float2(-snB.x, -snB.y), nsnC = make_float2(-snC.x, -snC.y);
          const int t = tg * TPG + i;
#pragma unroll
          for (int r = 0; r < R; ++r) {
            // elements (n, r) for n = 4kk2 + e; .x holds pair k0 (e = 0, 1), .y pair k0+1 (e = 2, 3)
            const float4 bq = *reinterpret_cast<const float4*>(&s_biasT[0][r][4 * kk2]);
            float2 b0 = make_float2(bf_at(bw[i], 0 * R + r), bf_at(bw[i], 2 * R + r));
            float2 b1 = make_float2(bf_at(bw[i], 1 * R + r), bf_at(bw[i], 3 * R + r));
            b0 = add2(b0, make_float2(bq.x, bq.z));
            b1 = add2(b1, make_float2(bq.y, bq.w));
            // Rot(-Phi) = [[cos, sin], [-sin, cos]]
            const float2 bt0 = fma2(csB, b0, mul2(snB, b1)), bt1 = fma2(csB, b1, mul2(nsnB, b0));
            const uint32_t o = tile_off((uint32_t)(t * R + r), 4u * kk2, 64u);
            sts64(opb + K::kOpBt + o, pack_f16(bt0.x, bt1.x), pack_f16(bt0.y, bt1.y));
            if constexpr (!SO) {
              const float4 cq = *reinterpret_cast<const float4*>(&s_biasT[1][r][4 * kk2]);
              float2 c0 = make_float2(bf_at(cw[i], 0 * R + r), bf_at(cw[i], 2 * R + r));
              float2 c1 = make_float2(bf_at(cw[i], 1 * R + r), bf_at(cw[i], 3 * R + r));
              c0 = add2(c0, make_float2(cq.x, cq.z));
              c1 = add2(c1, make_float2(cq.y, cq.w));
              const float2 ct0 = fma2(csC, c0, mul2(snC, c1)), ct1 = fma2(csC, c1, mul2(nsnC, c0));
              sts64(opb + K::kOpCt + o, pack_f16(ct0.x, ct1.x), pack_f16(ct0.y, ct1.y));
            }
          }
        }
      }
      // 6. w X (fp16, scaled) and X as the [(token, rank)][p] bf16 operand
#pragma unroll
      for (int j = 0; j < kXItems; ++j) {
        const int it = tid + kProThreads * j;
        if constexpr (R == 1) {
          // the raw tile is already 128-byte swizzled [token][p]: same offsets
          const uint32_t row = (uint32_t)it >> 3;
          const float w = sc.wend[row] * sigX;
          const uint4 v = xv[j][0];
          if constexpr (!SO) sts128(opb + K::kOpXo + (uint32_t)it * 16u, v);
          sts128(opb + K::kOpXw + (uint32_t)it * 16u,
                 make_uint4(pack_f16(w * bf_lo(v.x), w * bf_hi(v.x)),
                            pack_f16(w * bf_lo(v.y), w * bf_hi(v.y)),
                            pack_f16(w * bf_lo(v.z), w * bf_hi(v.z)),
                            pack_f16(w * bf_lo(v.w), w * bf_hi(v.w))));
        } else {
          const int sx = it / (kP / 4), pb = it % (kP / 4);
          uint32_t wv[2 * R];
#pragma unroll
          for (int q = 0; q < kXVec; ++q) {
            wv[4 * q] = xv[j][q].x; wv[4 * q + 1] = xv[j][q].y;
            wv[4 * q + 2] = xv[j][q].z; wv[4 * q + 3] = xv[j][q].w;
          }
          const float w = sc.wend[sx] * sigX;
#pragma unroll
          for (int r = 0; r < R; ++r) {
            float v4[4];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) v4[q4] = bf_at(wv, q4 * R + r);
            const uint32_t o = sw128((uint32_t)(sx * R + r), 4u * pb);
            if constexpr (!SO) sts64(opb + K::kOpXo + o, pack_bf16(v4[0], v4[1]), pack_bf16(v4[2], v4[3]));
            sts64(opb + K::kOpXw + o, pack_f16(w * v4[0], w * v4[1]), pack_f16(w * v4[2], w * v4[3]));
          }
        }
      }
      // 7. S = Ct Bt^T and D = Bt^T (w X) of this chunk into TMEM set s (free
      // since the core released slot s), then publish the slot to the core
      ptx::fence_proxy_async_smem();
      ptx::named_bar_sync(kBarPro, kProThreads);
      // (S and D from two warps, so that the two issue sequences overlap)
      if ((!SO && tid == kSTid) || tid == kDTid) {
        const uint32_t tset = tmem + (uint32_t)s * kTmemSlot;
        ptx::tc_fence_after_sync();
        if (tid == kDTid) {
          const Desc dBm = make_desc(opb + K::kOpBt, 64u * 128u);
          const Desc dXw = make_desc(opb + K::kOpXw, 64u * 128u);
#pragma unroll
          for (int kk = 0; kk < kQR / 16; ++kk)
            ptx::mma_bf16_ss(tset + kColD, desc_at(dBm, koff_mn(kk)), desc_at(dXw, koff_mn(kk)), kIdD,
                             kk > 0);
        } else {
          const Desc dBk = make_desc(opb + K::kOpBt, 16u), dCk = make_desc(opb + K::kOpCt, 16u);
#pragma unroll
          for (int kk = 0; kk < NS / 16; ++kk)
            ptx::mma_bf16_ss(tset + kColS, desc_at(dCk, koff_k(kk, 64)), desc_at(dBk, koff_k(kk, 64)),
                             kIdS, kk > 0);
        }
        ptx::mma_commit(&bar_acc_full[s]);
        if (tid == kDTid) ptx::mbar_arrive(&bar_op_full[s]);
      }
      if (!has_next) break;
      sch.next(p);  // = nxt, recomputed rather than kept live across the body
    }
    // on an early exit, let an issued load land before the CTA ends
    if (tid == kTmaTid && inflight >= 0) ptx::mbar_wait(&bar_raw_full, (uint32_t)inflight, kWaitNs);
  } else {
    // ============================================================ core (+ MMA issue)
    const int ct = tid - kProThreads;  // 0..127
    const int quad = warp & 3;         // TMEM lane quadrant of this warp
    const int half = (warp - kProWarps) >> 2;  // which 32-column half of the tiles it takes
    const int cwarp = warp - kProWarps;        // 0 .. kCoreWarps - 1
    float hreg[HR];
    float h_inv_prev = 1.f;
    float dsum = 0.f;  // log2 decay accumulated over the unit (state-only pass)
    // state element (n, cb + j) of this thread's 16-column block `blk` is hreg[16 blk + j]
    auto hpos = [&](int blk, uint32_t& n, uint32_t& cb) {
      if constexpr (NS == 128) {
        n = (uint32_t)(32 * quad + lane);  // M=128 accumulator layout: lane = row
        cb = 32u * half + 16u * blk;
      } else {
        n = (uint32_t)(16 * quad + (lane & 15));  // M=64 layout: 16 rows per quadrant
        cb = 32u * half + 16u * (lane >> 4);
      }
    };
    // fp16 copy of sigma * hreg into the state tile (operand of the next Yoff)
    auto write_hcopy = [&](float h_sig) {
      const float2 hs2 = make_float2(h_sig, h_sig);
#pragma unroll
      for (int blk = 0; blk < HR / 16; ++blk) {
        uint32_t n, cb;
        hpos(blk, n, cb);
        uint32_t wv[8];
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          const float2 v = mul2(hs2, make_float2(hreg[16 * blk + j], hreg[16 * blk + j + 1]));
          wv[j >> 1] = pack_f16(v.x, v.y);
        }
        sts128(sbase + K::kH + sw128(n, cb), make_uint4(wv[0], wv[1], wv[2], wv[3]));
        sts128(sbase + K::kH + sw128(n, cb + 8u), make_uint4(wv[4], wv[5], wv[6], wv[7]));
      }
    };
    // Yoff = Ct H of chunk g into set g & 1 (this thread's next commit, after
    // the chunk's Y, covers it)
    auto issue_yoff = [&](int g) {
      const int s = g & 1;
      const uint32_t tset = tmem + (uint32_t)s * kTmemSlot;
      const uint32_t opb = sbase + K::kOp0 + (uint32_t)s * K::kOpBytes;
      const Desc dCk = make_desc(opb + K::kOpCt, 16u), dH = make_desc(sbase + K::kH, (uint32_t)NS * 128u);
      ptx::tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < NS / 16; ++kk)
        ptx::mma_bf16_ss(tset + kColYo, desc_at(dCk, koff_k(kk, 64)), desc_at(dH, koff_mn(kk)), kIdYo,
                         kk > 0);
    };
    // State entering unit u: the given explicit-frame state (the unit's local
    // angle frame starts at zero, so no rotation) or zero; in the full pass its
    // fp16 copy feeds the unit's first Yoff.
    auto enter_unit = [&](int64_t u) {
      dsum = 0.f;
      if (p.ws_hin) {
        const float* src = p.ws_hin + u * (int64_t)NS * kP;
        float m = 0.f;
#pragma unroll
        for (int blk = 0; blk < HR / 16; ++blk) {
          uint32_t n, cb;
          hpos(blk, n, cb);
          const float4* q4 = reinterpret_cast<const float4*>(src + (int64_t)n * kP + cb);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float4 v = q4[j];
            hreg[16 * blk + 4 * j] = v.x;
            hreg[16 * blk + 4 * j + 1] = v.y;
            hreg[16 * blk + 4 * j + 2] = v.z;
            hreg[16 * blk + 4 * j + 3] = v.w;
            m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
          }
        }
        if constexpr (!SO) {
          m = warp_max(m);
          if (lane == 0) s_hred[cwarp] = m;
          ptx::named_bar_sync(kBarCore, kCoreThreads);
          float mm = 0.f;
#pragma unroll
          for (int w = 0; w < kCoreWarps; ++w) mm = fmaxf(mm, s_hred[w]);
          float h_sig;
          pow2_scale(mm, &h_sig, &h_inv_prev);
          write_hcopy(h_sig);
          ptx::fence_proxy_async_smem();
          ptx::tc_fence_before_sync();
          ptx::named_bar_sync(kBarCore, kCoreThreads);
        }
      } else {
#pragma unroll
        for (int i = 0; i < HR; ++i) hreg[i] = 0.f;
      }
    };
    Sched sch;
    sch.start(blockIdx.x, p);
    enter_unit(sch.unit);
    if (!SO && p.ws_hin && ct == 0 && wait_or_abort(&bar_op_full[0], 0u, &abort_flag, p.status))
      issue_yoff(0);
    for (int g = 0;; ++g) {
      const int b = sch.b, h = sch.h;
      const int c = sch.c, s = g & 1;
      const bool first = c == sch.c_begin, last = c == sch.c_end - 1;
      const bool has_next = sch.c + 1 < sch.c_end || sch.unit + (int)gridDim.x < p.nunits;
      const SlotScalars<KP>& sc = ss[s];
      const uint32_t tset = tmem + (uint32_t)s * kTmemSlot;
      if (ct == 0)
        s_go[1] = wait_or_abort(&bar_acc_full[s], (uint32_t)((g >> 1) & 1), &abort_flag, p.status)
                      ? 1 : 0;
      ptx::named_bar_sync(kBarCore, kCoreThreads);
      if (!s_go[1]) break;
      ptx::tc_fence_after_sync();
      const float invB = sc.invB, invC = sc.invC, invX = sc.invX;
      if constexpr (!SO) {
        // ---- masked scores: thread -> row a, 16 consecutive columns per block
        const int a = 16 * quad + (lane & 15);
        const int t = a / R;
        const float einv = (float)((int)((__float_as_uint(invB * invC) >> 23) & 0xffu) - 127);
        const float lt = sc.lam2[t] + einv;
        const float gdiag = sc.gam[t] * (invB * invC);
        // this warp's 32-column block; skip it when its 16 rows x 32 columns lie
        // wholly above the diagonal
        for (int blk = half; blk == half; ++blk) {
          if ((32 * blk) / R > (16 * quad + 15) / R) continue;
          uint32_t sv[16];
          ptx::tmem_ld16_16x32bx2<16>(tset + kColS + ((uint32_t)(32 * quad) << 16) + 32u * blk, sv);
          ptx::tmem_ld_wait(sv);
          const int c0 = 32 * blk + 16 * (lane >> 4);
          if (c0 / R > t) continue;
          constexpr int NT = 16 / R;  // distinct tokens among the 16 columns
          const int s0 = c0 / R;
          float lsv[NT], wpv[NT];  // s0 is a multiple of NT >= 4: 16-byte aligned
#pragma unroll
          for (int u = 0; u < NT; u += 4) {
            *reinterpret_cast<float4*>(&lsv[u]) = *reinterpret_cast<const float4*>(&sc.lam2[s0 + u]);
            *reinterpret_cast<float4*>(&wpv[u]) = *reinterpret_cast<const float4*>(&sc.wp[s0 + u]);
          }
          uint32_t ph_[8], pl_[8];
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            // two columns at a time (packed fp32 pairs; same roundings as scalar)
            const int u0 = j / R, u1 = (j + 1) / R;
            const float2 dl = sub2(make_float2(lt, lt), make_float2(lsv[u0], lsv[u1]));
            const float2 mo = mul2(make_float2(ex2(dl.x), ex2(dl.y)), make_float2(wpv[u0], wpv[u1]));
            const float m0 = (s0 + u0 < t) ? mo.x : ((s0 + u0 == t) ? gdiag : 0.f);
            const float m1 = (s0 + u1 < t) ? mo.y : ((s0 + u1 == t) ? gdiag : 0.f);
            const float2 v2 = mul2(make_float2(m0, m1),
                                   make_float2(__uint_as_float(sv[j]), __uint_as_float(sv[j + 1])));
            const uint32_t hw = pack_bf16(v2.x, v2.y);
            ph_[j >> 1] = hw;
            const float2 lo = sub2(v2, make_float2(bf_lo(hw), bf_hi(hw)));
            pl_[j >> 1] = pack_bf16(lo.x, lo.y);
          }
          const uint32_t o0 = sw128((uint32_t)a, (uint32_t)c0);
          const uint32_t o1 = sw128((uint32_t)a, (uint32_t)c0 + 8u);
          sts128(sbase + K::kPh + o0, make_uint4(ph_[0], ph_[1], ph_[2], ph_[3]));
          sts128(sbase + K::kPh + o1, make_uint4(ph_[4], ph_[5], ph_[6], ph_[7]));
          sts128(sbase + K::kPl + o0, make_uint4(pl_[0], pl_[1], pl_[2], pl_[3]));
          sts128(sbase + K::kPl + o1, make_uint4(pl_[4], pl_[5], pl_[6], pl_[7]));
        }
        ptx::fence_proxy_async_smem();
        ptx::named_bar_sync(kBarCore, kCoreThreads);
        if (ct == 0) {
          // Y = P X (P = high + low parts) of this chunk
          const uint32_t opb = sbase + K::kOp0 + (uint32_t)s * K::kOpBytes;
          const Desc dPh = make_desc(sbase + K::kPh, 16u), dPl = make_desc(sbase + K::kPl, 16u);
          const Desc dX = make_desc(opb + K::kOpXo, 64u * 128u);
          ptx::tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < kQR / 16; ++kk)
            ptx::mma_bf16_ss(tset + kColY, desc_at(dPh, koff_k(kk, 64)), desc_at(dX, koff_mn(kk)),
                             kIdY, kk > 0);
#pragma unroll
          for (int kk = 0; kk < kQR / 16; ++kk)
            ptx::mma_bf16_ss(tset + kColY, desc_at(dPl, koff_k(kk, 64)), desc_at(dX, koff_mn(kk)),
                             kIdY, 1u);
          ptx::mma_commit(&bar_y_full[s]);
        }
      }
      // ---- state: H = exp(Lam_end) H + D / (sigma_B sigma_X)
      float hmax = 0.f;
      {
        const float2 e2 = make_float2(sc.eLend, sc.eLend);
        const float iBX = invB * invX;
        const float2 i2 = make_float2(iBX, iBX);
#pragma unroll
        for (int blk = 0; blk < HR / 16; ++blk) {
          uint32_t d[16];
          if constexpr (NS == 128) {
            ptx::tmem_ld16(tset + kColD + ((uint32_t)(32 * quad) << 16) + 32u * half + 16u * blk, d);
          } else {
            ptx::tmem_ld16_16x32bx2<16>(tset + kColD + ((uint32_t)(32 * quad) << 16) + 32u * half, d);
          }
          ptx::tmem_ld_wait(d);
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            float2 hv = mul2(e2, make_float2(hreg[16 * blk + j], hreg[16 * blk + j + 1]));
            hv = fma2(i2, make_float2(__uint_as_float(d[j]), __uint_as_float(d[j + 1])), hv);
            hreg[16 * blk + j] = hv.x;
            hreg[16 * blk + j + 1] = hv.y;
            if constexpr (!SO) hmax = fmaxf(hmax, fmaxf(fabsf(hv.x), fabsf(hv.y)));
          }
        }
      }
      if constexpr (SO) dsum += sc.lamend2;
      bool next_issued = false;
      if constexpr (!SO) {
        hmax = warp_max(hmax);
        if (lane == 0) s_hred[cwarp] = hmax;
        // Y (and this chunk's Yoff, which read the previous state copy) complete;
        // the output staging tile is free again
        if (ct == 0) {
          s_go[1] = wait_or_abort(&bar_y_full[s], (uint32_t)((g >> 1) & 1), &abort_flag, p.status)
                        ? 1 : 0;
          ptx::tma_store_wait_read<0>();
        }
        ptx::named_bar_sync(kBarCore, kCoreThreads);
        if (!s_go[1]) break;
        ptx::tc_fence_after_sync();
        float h_inv = h_inv_prev;
        if (!last) {
          // fp16 copy of the new state for the next chunk's Ct H product
          float m = 0.f;
#pragma unroll
          for (int w = 0; w < kCoreWarps; ++w) m = fmaxf(m, s_hred[w]);
          float h_sig;
          pow2_scale(m, &h_sig, &h_inv);
          write_hcopy(h_sig);
          ptx::fence_proxy_async_smem();
          ptx::tc_fence_before_sync();
          ptx::named_bar_sync(kBarCore, kCoreThreads);
          // the next chunk's Yoff, if its operands are ready already
          if (ct == 0 &&
              ptx::mbar_try_wait(&bar_op_full[(g + 1) & 1], (uint32_t)(((g + 1) >> 1) & 1))) {
            issue_yoff(g + 1);
            next_issued = true;
          }
        }
        // ---- outputs: y = Y + exp(Lam_t) Yoff
        {
          const int a = 16 * quad + (lane & 15);
          const float el = sc.eL[a / R] * (invC * h_inv_prev);
          const bool has_yoff = !first || p.ws_hin != nullptr;
          for (int blk = half; blk == half; ++blk) {
            uint32_t yv[16];
            const uint32_t ta = ((uint32_t)(32 * quad) << 16) + 32u * blk;
            ptx::tmem_ld16_16x32bx2<16>(tset + kColY + ta, yv);
            ptx::tmem_ld_wait(yv);
            const int c0 = 32 * blk + 16 * (lane >> 4);  // first p of this thread
            float y[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) y[j] = __uint_as_float(yv[j]);
            if (has_yoff) {
              // a unit that starts from a zero state has no Yoff for its first
              // chunk (that accumulator was not written)
              uint32_t yo[16];
              ptx::tmem_ld16_16x32bx2<16>(tset + kColYo + ta, yo);
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
              const uint32_t o0 = sw128((uint32_t)a, (uint32_t)c0);
              const uint32_t o1 = sw128((uint32_t)a, (uint32_t)c0 + 8u);
              sts128(sbase + K::kYs + o0, make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]),
                                                     pack_bf16(y[4], y[5]), pack_bf16(y[6], y[7])));
              sts128(sbase + K::kYs + o1,
                     make_uint4(pack_bf16(y[8], y[9]), pack_bf16(y[10], y[11]),
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
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before_sync();
        ptx::named_bar_sync(kBarCore, kCoreThreads);
        if (ct == 0) {
          ptx::tma_store_4d(&tm_y, smem + K::kYs, 0, h, c * Q, b);
          ptx::tma_store_commit();
        }
        h_inv_prev = h_inv;
      }
      if (last) {
        if constexpr (SO) {
          // the unit's local end state and its (log2 decay, angle) totals
          float* dst = p.ws_state + sch.unit * (int64_t)NS * kP;
#pragma unroll
          for (int blk = 0; blk < HR / 16; ++blk) {
            uint32_t n, cb;
            hpos(blk, n, cb);
            float4* q4 = reinterpret_cast<float4*>(dst + (int64_t)n * kP + cb);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              q4[j] = make_float4(hreg[16 * blk + 4 * j], hreg[16 * blk + 4 * j + 1],
                                  hreg[16 * blk + 4 * j + 2], hreg[16 * blk + 4 * j + 3]);
          }
          float* sd = p.ws_scal + sch.unit * (int64_t)(1 + KP);
          if (ct == 0) sd[0] = dsum;
          if (ct < KP) sd[1 + ct] = sc.fang[ct];
        } else if (c == nC - 1 && p.final_state) {
          // final state of the sequence, explicit frame: h = Rot(Phi_{L-1}) g
          float* fs = p.final_state + ((int64_t)b * p.heads + h) * NS * kP;
#pragma unroll
          for (int blk = 0; blk < HR / 16; ++blk) {
            uint32_t n, cb;
            hpos(blk, n, cb);
            // the carried angle is wrapped to [-pi, pi]: the fast sincos is
            // accurate there (and keeps the accurate version's large slow path
            // out of the loop's code)
            float sn, cs;
            __sincosf(sc.fang[n >> 1], &sn, &cs);
            const bool odd = n & 1;
            float o[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float hv = hreg[16 * blk + j];
              const float other = __shfl_xor_sync(0xffffffffu, hv, 1);
              // even row: c g0 - s g1 ; odd row: s g0 + c g1
              o[j] = odd ? fmaf(sn, other, cs * hv) : fmaf(-sn, other, cs * hv);
            }
            float4* dst = reinterpret_cast<float4*>(fs + (int64_t)n * kP + cb);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[j] = make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
          }
        }
        if (has_next) enter_unit(sch.unit + (int)gridDim.x);
      }
      ptx::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bar_slot_free[s]);
      if constexpr (!SO) {
        // the next chunk's Yoff if it could not go out above
        const bool want_yoff = has_next && (!last || p.ws_hin != nullptr);
        if (ct == 0 && want_yoff && !next_issued &&
            wait_or_abort(&bar_op_full[(g + 1) & 1], (uint32_t)(((g + 1) >> 1) & 1), &abort_flag,
                          p.status))
          issue_yoff(g + 1);
      }
      if (!has_next) break;
      sch.next(p);
    }
    if (ct == 0) ptx::tma_store_wait_all<0>();
  }

  // ---------------------------------------------------------------- teardown
  ptx::tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpTmem) {
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

// x / out as a 4-D tensor {P*R, H, L, b}; the box is one head's chunk.
bool make_act_map(CUtensorMap* m, const void* ptr, const ScanArgs& a) {
  const uint64_t PR = (uint64_t)a.P * a.R;
  cuuint64_t dims[4] = {PR, (cuuint64_t)a.H, (cuuint64_t)a.L, (cuuint64_t)a.batch};
  cuuint64_t strides[3] = {PR * 2, PR * 2 * a.H, PR * 2 * a.H * a.L};
  cuuint32_t box[4] = {(cuuint32_t)PR, 1, (cuuint32_t)a.Q, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, ptr, dims, strides, box,
                a.R == 1 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

// B / C [b, L, G, N, R] as a 5-D tensor {d0, N*R/d0, G, L, b} with d0 <= 256.
bool make_bc_map(CUtensorMap* m, const void* ptr, const ScanArgs& a) {
  const uint64_t NR = (uint64_t)a.N * a.R;
  const uint64_t d0 = NR < 256 ? NR : 256, d1 = NR / d0;
  cuuint64_t dims[5] = {d0, d1, (cuuint64_t)a.G, (cuuint64_t)a.L, (cuuint64_t)a.batch};
  cuuint64_t strides[4] = {d0 * 2, NR * 2, NR * 2 * a.G, NR * 2 * a.G * a.L};
  cuuint32_t box[5] = {(cuuint32_t)d0, (cuuint32_t)d1, 1, (cuuint32_t)a.Q, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, ptr, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_NONE);
}

// theta [b, L, G, N/2] fp32 as {N/2, G, L, b}.
bool make_theta_map(CUtensorMap* m, const float* ptr, const ScanArgs& a) {
  const uint64_t KP = (uint64_t)a.N / 2;
  cuuint64_t dims[4] = {KP, (cuuint64_t)a.G, (cuuint64_t)a.L, (cuuint64_t)a.batch};
  cuuint64_t strides[3] = {KP * 4, KP * 4 * a.G, KP * 4 * a.G * a.L};
  cuuint32_t box[4] = {(cuuint32_t)KP, 1, (cuuint32_t)a.Q, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ptr, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_NONE);
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

template <int R, int NS, bool SO>
cudaError_t launch_pass(const CUtensorMap* maps, const TcParams& p, int64_t units, cudaStream_t s) {
  constexpr uint32_t smem = Cfg<R, NS>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(scan_tc_kernel<R, NS, SO>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int sms = num_sms();
  if (sms <= 0) return cudaErrorInvalidValue;
  const unsigned grid = (unsigned)(units < sms ? units : sms);
  scan_tc_kernel<R, NS, SO><<<grid, kThreads, smem, s>>>(maps[0], maps[1], maps[2], maps[3],
                                                          maps[4], p);
  return cudaGetLastError();
}

template <int R, int NS>
cudaError_t launch_rn(const ScanArgs& a, unsigned int* status, cudaStream_t s) {
  CUtensorMap maps[5];
  if (!make_bc_map(&maps[0], a.B, a) || !make_bc_map(&maps[1], a.C, a) ||
      !make_theta_map(&maps[2], a.theta, a) || !make_act_map(&maps[3], a.x, a) ||
      !make_act_map(&maps[4], a.out, a))
    return cudaErrorInvalidValue;
  TcParams p;
  p.dt = a.dt; p.A = a.A; p.lam = a.lam;
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
  if (pl.nseg <= 1) return launch_pass<R, NS, false>(maps, p, nseq, s);
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
  cudaError_t e = launch_pass<R, NS, true>(maps, p, units, s);
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
    e = launch_pass<R, NS, false>(maps, p, units, s);
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
