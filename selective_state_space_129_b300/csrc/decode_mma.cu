// Decode of the Mamba-3 scan at MIMO rank R = 4 (bf16 activations, P = 64)
// with the rank-R update on the tensor cores: one token per call, and K
// consecutive tokens per call with the state held on chip between them.
//
// For every (batch, head) a token's step is (Prop. 1 and the rotation, sec. 4.1
// and 4.2 of "MAMBA-3: IMPROVED SEQUENCE MODELING USING STATE SPACE PRINCIPLES"
// (aipaper.cc); MIMO rank R, sec. 3 of "Mamba-3: Improved Sequence Modeling
// using State Space Principles" (papernotes.org)):
//   h' = alpha Rot(Delta theta) (h + beta_hat (B_prev + bias) x_prev^T) + gamma (B + bias) x^T
//   y  = (C + bias)^T h'
// The rotation acts on rows, so alpha Rot (beta_hat (B_prev + bias) x_prev^T)
// = (alpha Rot beta_hat (B_prev + bias)) x_prev^T, and
//   h' = alpha Rot h + U X^T,  U = [alpha Rot beta_hat (B_prev + bias) | gamma (B + bias)] (N x 2R),
//                              X = [x_prev | x] (P x 2R).
// U X^T is a rank-2R (= 8) product: it runs as mma.sync m16n8k8 (bf16 in,
// fp32 accumulate), with U split into bf16 high and low parts (U ~ hi + lo to
// about 16 bits) against the exact bf16 X. An MMA tile is 8 rotating row
// pairs x 8 state columns: MMA row i is state row 2(k0 + i) and row i + 8 is
// state row 2(k0 + i) + 1, so that every thread's accumulator holds both rows
// of a pair (the rotation stays in the thread). Warp w owns state columns
// 8w .. 8w + 7 over all rows, held in its registers, so its partial y needs
// only a reduction across its own lanes.
//
// One token is bound by HBM traffic (the fp32 state is read and written once):
// a persistent kernel (two 256-thread CTAs per SM) streams the (b, h) units
// through two stages of shared memory, the state by TMA with the 128-byte
// swizzle (so that the MMA layout's 8 rows x 8 columns loads are free of bank
// conflicts), the token's activations by bulk copies. K tokens read and write
// the state once for all K: one CTA per (b, h) loads the state and the K
// tokens' activations, builds the tables of a window of tokens in one
// parallel pass (in the shared memory the state came through), and runs the
// window's tokens back to back with no barrier between them.
//
// Every wait is bounded; an expired wait sets the status word and the CTA
// leaves at the next barrier without writing the state.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace m3 {
namespace {

constexpr int kMThreads = 256;
constexpr int kMR = 4;   // rank
constexpr int kMP = 64;  // head dim: 8 warps x 8 columns
constexpr int kMStages = 2;
constexpr uint64_t kMWaitNs = 2000000000ull;  // 2 s per wait
constexpr int kMaxNT = 8;  // N up to 128: 16 state rows per MMA row tile
constexpr uint32_t kPairWords = 12;  // U table words per row pair (8 used; padded off bank conflicts)
constexpr size_t kMSmemMax = 112 * 1024;  // two CTAs per SM

__host__ __device__ constexpr uint32_t up16m(uint64_t v) { return (uint32_t)((v + 15) & ~15ull); }
__host__ __device__ constexpr uint32_t up1k(uint64_t v) { return (uint32_t)((v + 1023) & ~1023ull); }

// Tables of one token: U high and low parts [N/2 pairs][kPairWords] (row 2k at
// words 0-3, row 2k + 1 at words 4-7, each as 2R = 8 bf16), C + bias [N][R]
// fp32, alpha (cos, sin) [N/2].
__host__ __device__ inline uint32_t mma_table_bytes(int64_t N) {
  return (uint32_t)(2 * (N / 2) * kPairWords * 4 + N * kMR * 4 + (N / 2) * 8);
}

struct TokTab {
  uint32_t* Uh;
  uint32_t* Ul;
  float* cd;
  float2* rd;
};

__device__ __forceinline__ TokTab tok_tab(uint8_t* base, int N) {
  TokTab T;
  T.Uh = reinterpret_cast<uint32_t*>(base);
  T.Ul = T.Uh + (N / 2) * kPairWords;
  T.cd = reinterpret_cast<float*>(T.Ul + (N / 2) * kPairWords);
  T.rd = reinterpret_cast<float2*>(T.cd + N * kMR);
  return T;
}

// Entry (row pair kq, rank r) of a token's tables. B, C [N][R] and the biases
// are in shared memory; Bp (the previous token's B) and the biases may be null.
__device__ __forceinline__ void table_entry(const TokTab& T, int kq, int r, float alpha,
                                            float gamma, float bhat, float phi,
                                            const __nv_bfloat16* B, const __nv_bfloat16* Bp,
                                            const __nv_bfloat16* C, const float* bb,
                                            const float* cb) {
  float sn, cs;
  __sincosf(wrap_angle(phi), &sn, &cs);
  const float ac = alpha * cs, as = alpha * sn;
  const int i0 = 2 * kq * kMR + r, i1 = i0 + kMR;  // (row 2kq, r), (row 2kq + 1, r)
  const float bb0 = bb ? bb[i0] : 0.f, bb1 = bb ? bb[i1] : 0.f;
  const float cb0 = cb ? cb[i0] : 0.f, cb1 = cb ? cb[i1] : 0.f;
  float u0 = 0.f, u1 = 0.f;
  if (Bp != nullptr) {
    const float q0 = bhat * (ld_act(Bp + i0) + bb0), q1 = bhat * (ld_act(Bp + i1) + bb1);
    u0 = fmaf(ac, q0, -as * q1);
    u1 = fmaf(as, q0, ac * q1);
  }
  const float g0 = gamma * (ld_act(B + i0) + bb0), g1 = gamma * (ld_act(B + i1) + bb1);
  // U row 2kq: [u0 | g0] at bf16 index r and R + r; row 2kq + 1 eight further
  __nv_bfloat16* Uh16 = reinterpret_cast<__nv_bfloat16*>(T.Uh) + kq * 2 * kPairWords;
  __nv_bfloat16* Ul16 = reinterpret_cast<__nv_bfloat16*>(T.Ul) + kq * 2 * kPairWords;
  const float v[4] = {u0, g0, u1, g1};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(v[q]);
    Uh16[q * kMR + r] = hi;
    Ul16[q * kMR + r] = __float2bfloat16_rn(v[q] - __bfloat162float(hi));
  }
  T.cd[i0] = ld_act(C + i0) + cb0;
  T.cd[i1] = ld_act(C + i1) + cb1;
  if (r == 0) T.rd[kq] = make_float2(ac, as);
}

__device__ __forceinline__ void mma_bf16_16x8x8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5}, {%6}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b));
}

__device__ __forceinline__ uint32_t bf16_pair(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Byte offset of state element (n, col) in shared memory: column half, row n
// (128 bytes), 16-byte chunk XOR the row's low three bits (the TMA 128B swizzle).
__device__ __forceinline__ uint32_t st_off(uint32_t half_bytes, uint32_t n, uint32_t col) {
  const uint32_t cl = col & 31u;
  return (col >> 5) * half_bytes + n * 128u + ((((cl >> 2) ^ n) & 7u) << 4) + (cl & 3u) * 4u;
}

// The warp's columns p0, p0 + 1 (p0 = 8 warp + 2 tq) of rows 2kq, 2kq + 1
// (kq = 8 rt + g) from the swizzled state in shared memory into registers.
template <int NT>
__device__ __forceinline__ void load_state(float2 (&h0)[NT], float2 (&h1)[NT], const uint8_t* st,
                                           uint32_t half, int g, int p0) {
  // row 2kq = 2g + 16 rt: the swizzle phase (row & 7) is the same for every rt
  const uint8_t* r0 = st + st_off(half, 2u * g, (uint32_t)p0);
  const uint8_t* r1 = st + st_off(half, 2u * g + 1u, (uint32_t)p0);
#pragma unroll
  for (int rt = 0; rt < NT; ++rt) {
    h0[rt] = *reinterpret_cast<const float2*>(r0 + rt * 16 * 128);
    h1[rt] = *reinterpret_cast<const float2*>(r1 + rt * 16 * 128);
  }
}

// X fragment of the warp: X[p = 8 warp + g][k = 2 tq, 2 tq + 1], k < R from
// x_prev (zero when xp is null), else from x; both [P][R] bf16.
__device__ __forceinline__ uint32_t x_fragment(const uint8_t* x, const uint8_t* xp, int warp,
                                               int g, int tq) {
  const int pcol = 8 * warp + g;
  if (tq < 2) {
    if (xp == nullptr) return 0u;
    return reinterpret_cast<const uint32_t*>(xp)[pcol * (kMR / 2) + tq];
  }
  return reinterpret_cast<const uint32_t*>(x)[pcol * (kMR / 2) + (tq & 1)];
}

// One token on the warp's 8 columns: h' = alpha Rot h + U X^T (in registers),
// y = C^T h' summed over the warp and stored as bf16 at yw (the warp's 32
// outputs, [8 columns][R]); with STORE the new state rows also go to gst
// (the unit's [N][P] fp32 state in global memory).
template <int NT, bool STORE>
__device__ __forceinline__ void token_step(float2 (&h0)[NT], float2 (&h1)[NT], const TokTab& T,
                                           uint32_t bx, float* gst, __nv_bfloat16* yw, int g,
                                           int tq, int p0) {
  float2 yv[kMR];  // (y[p0][r], y[p0 + 1][r])
#pragma unroll
  for (int r = 0; r < kMR; ++r) yv[r] = make_float2(0.f, 0.f);
#pragma unroll
  for (int rt = 0; rt < NT; ++rt) {
    const int kq = 8 * rt + g;  // this thread's row pair
    float dacc[4] = {0.f, 0.f, 0.f, 0.f};
    mma_bf16_16x8x8(dacc, T.Uh[kq * kPairWords + tq], T.Uh[kq * kPairWords + 4 + tq], bx);
    mma_bf16_16x8x8(dacc, T.Ul[kq * kPairWords + tq], T.Ul[kq * kPairWords + 4 + tq], bx);
    const float2 rot = T.rd[kq];
    const float2 ac2 = make_float2(rot.x, rot.x), as2 = make_float2(rot.y, rot.y);
    const float2 nas2 = make_float2(-rot.y, -rot.y);
    // rows 2kq, 2kq + 1: alpha [[c, -s], [s, c]] (h0, h1) + U X^T
    const float2 r0 = ptx::fma2(ac2, h0[rt], ptx::fma2(nas2, h1[rt], make_float2(dacc[0], dacc[1])));
    const float2 r1 = ptx::fma2(as2, h0[rt], ptx::fma2(ac2, h1[rt], make_float2(dacc[2], dacc[3])));
    h0[rt] = r0;
    h1[rt] = r1;
    if (STORE) {
      *reinterpret_cast<float2*>(gst + (int64_t)(2 * kq) * kMP + p0) = r0;
      *reinterpret_cast<float2*>(gst + (int64_t)(2 * kq + 1) * kMP + p0) = r1;
    }
    const float4 ce = *reinterpret_cast<const float4*>(T.cd + 2 * kq * kMR);
    const float4 co = *reinterpret_cast<const float4*>(T.cd + (2 * kq + 1) * kMR);
    const float cev[4] = {ce.x, ce.y, ce.z, ce.w}, cov[4] = {co.x, co.y, co.z, co.w};
#pragma unroll
    for (int r = 0; r < kMR; ++r)
      yv[r] = ptx::fma2(make_float2(cev[r], cev[r]), r0,
                        ptx::fma2(make_float2(cov[r], cov[r]), r1, yv[r]));
  }
  // sum the eight values v[4c + r] = y[p0 + c][r] over the warp's row pairs
  // (the lanes that differ in g), halving the values at each step so that
  // lane (g, tq) ends with v[g] in full
  const bool b2 = (g & 4) != 0, b1 = (g & 2) != 0, b0 = (g & 1) != 0;
  float v[8], w[4], z[2];
#pragma unroll
  for (int r = 0; r < kMR; ++r) {
    v[r] = yv[r].x;
    v[kMR + r] = yv[r].y;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = b2 ? v[i] : v[i + 4];
    w[i] = (b2 ? v[i + 4] : v[i]) + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = b1 ? w[i] : w[i + 2];
    z[i] = (b1 ? w[i + 2] : w[i]) + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  const float t = (b0 ? z[1] : z[0]) + __shfl_xor_sync(0xffffffffu, b0 ? z[0] : z[1], 4);
  // v[g] is y[p0 + (g >> 2)][g & 3], at offset 8 tq + g of the warp's 32
  // outputs; even g stores itself and its odd neighbour as one bf16 pair
  const float t_next = __shfl_xor_sync(0xffffffffu, t, 4);
  if ((g & 1) == 0) *reinterpret_cast<uint32_t*>(yw + 8 * tq + g) = bf16_pair(t, t_next);
}

__device__ __forceinline__ void tma_state(uint8_t* dst, uint32_t half, const CUtensorMap* tm,
                                          uint64_t* bar, int u) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(ptx::smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(ptx::smem_addr(bar)), "r"(0), "r"(0), "r"(u)
      : "memory");
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(ptx::smem_addr(dst + half)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(ptx::smem_addr(bar)), "r"(32), "r"(0), "r"(u)
      : "memory");
}

// ------------------------------------------------------------- one token

// Byte offsets inside one stage: the state (two 128B-swizzled halves of 32
// columns, [N][32] fp32 each) first, then the token's blocks.
struct MmaLayout {
  uint32_t half, x, xp, B, Bp, C, th, bb, cb, dt, lm, act_bytes, bytes;
};

inline MmaLayout mma_layout(const DecodeArgs& a) {
  const uint64_t N = a.N, P = kMP, R = kMR;
  const bool prev = a.B_prev != nullptr;
  MmaLayout L{};
  L.half = (uint32_t)(N * 32 * 4);
  uint32_t o = 2 * L.half;
  const uint32_t act0 = o;
  L.x = o; o += up16m(P * R * 2);
  L.xp = o; o += prev ? up16m(P * R * 2) : 0u;
  L.B = o; o += up16m(N * R * 2);
  L.Bp = o; o += prev ? up16m(N * R * 2) : 0u;
  L.C = o; o += up16m(N * R * 2);
  L.th = o; o += up16m(N / 2 * 4);
  L.bb = o; o += a.B_bias ? up16m(N * R * 4) : 0u;
  L.cb = o; o += a.C_bias ? up16m(N * R * 4) : 0u;
  L.dt = o; o += 16;
  L.lm = o; o += 16;
  L.act_bytes = o - act0;
  L.bytes = up1k(o);
  return L;
}

// two stages, two table sets (alternating units), A [H]
inline size_t mma_smem_bytes(const DecodeArgs& a, const MmaLayout& L) {
  return 1024 + (size_t)kMStages * L.bytes + 2 * (size_t)mma_table_bytes(a.N) + 4 * (size_t)a.H;
}

template <int NT>
__global__ void __launch_bounds__(kMThreads, 2)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tm_state, DecodeArgs a, MmaLayout L,
                      int units) {
  extern __shared__ __align__(16) uint8_t dsm_raw[];
  // 1024-byte aligned (the 128B swizzle's atom); an offset from the array
  // keeps the accesses in the shared address space
  uint8_t* dsm = dsm_raw + ((1024u - (ptx::smem_addr(dsm_raw) & 1023u)) & 1023u);
  __shared__ uint64_t full[kMStages];
  __shared__ int abort_flag;
  const int N = (int)a.N, K2 = N / 2, H = (int)a.H;
  const int hpg = (int)(a.H / a.G);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;  // MMA group (row pair) and thread in group
  const int p0 = 8 * warp + 2 * tq;        // this thread's state columns p0, p0 + 1
  const uint32_t tbytes = mma_table_bytes(N);
  uint8_t* tables = dsm + (size_t)kMStages * L.bytes;
  float* sA = reinterpret_cast<float*>(tables + 2 * (size_t)tbytes);  // A [H]
  const bool has_prev = a.B_prev != nullptr;

  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < kMStages; ++s) ptx::mbar_init(&full[s], 1);
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&tm_state);
  }
  for (int i = tid; i < H; i += kMThreads) sA[i] = a.A[i];
  __syncthreads();

  // thread 0: stage unit u into stage s (the state by TMA, the rest by bulk copies)
  auto issue = [&](int u, int s) {
    const int b = u / H, h = u - b * H, gi = h / hpg;
    uint8_t* st = dsm + (size_t)s * L.bytes;
    uint64_t* bar = &full[s];
    const int64_t nr = (int64_t)N * kMR, pr = (int64_t)kMP * kMR;
    const int64_t bc = ((int64_t)b * a.G + gi) * nr;
    ptx::fence_proxy_async_smem();  // earlier reads of the stage come first
    ptx::mbar_arrive_expect_tx(bar, 2 * L.half + L.act_bytes);
    tma_state(st, L.half, &tm_state, bar, u);
    const __nv_bfloat16* X = static_cast<const __nv_bfloat16*>(a.x);
    ptx::bulk_load(st + L.x, X + (int64_t)u * pr, (uint32_t)(pr * 2), bar);
    if (has_prev)
      ptx::bulk_load(st + L.xp, static_cast<const __nv_bfloat16*>(a.x_prev) + (int64_t)u * pr,
                     (uint32_t)(pr * 2), bar);
    ptx::bulk_load(st + L.B, static_cast<const __nv_bfloat16*>(a.B) + bc, (uint32_t)(nr * 2), bar);
    if (has_prev)
      ptx::bulk_load(st + L.Bp, static_cast<const __nv_bfloat16*>(a.B_prev) + bc,
                     (uint32_t)(nr * 2), bar);
    ptx::bulk_load(st + L.C, static_cast<const __nv_bfloat16*>(a.C) + bc, (uint32_t)(nr * 2), bar);
    ptx::bulk_load(st + L.th, a.theta + ((int64_t)b * a.G + gi) * K2, (uint32_t)K2 * 4, bar);
    if (a.B_bias) ptx::bulk_load(st + L.bb, a.B_bias + (int64_t)h * nr, (uint32_t)nr * 4, bar);
    if (a.C_bias) ptx::bulk_load(st + L.cb, a.C_bias + (int64_t)h * nr, (uint32_t)nr * 4, bar);
    // dt, lambda of unit u: the aligned 16-byte window that holds them
    ptx::bulk_load(st + L.dt, a.dt + (u & ~3), 16u, bar);
    ptx::bulk_load(st + L.lm, a.lam + (u & ~3), 16u, bar);
  };
  int pending = 0;  // (thread 0) stages issued and not yet waited for
  if (tid == 0)
    for (int j = 0; j < kMStages; ++j) {
      const int u = blockIdx.x + j * (int)gridDim.x;
      if (u < units) {
        issue(u, j);
        ++pending;
      }
    }

  int k = 0;
  for (int u = blockIdx.x; u < units; u += gridDim.x, ++k) {
    const int s = k % kMStages;
    const uint8_t* stg = dsm + (size_t)s * L.bytes;
    const TokTab T = tok_tab(tables + (size_t)(k & 1) * tbytes, N);
    if (!ptx::mbar_wait(&full[s], (uint32_t)((k / kMStages) & 1), kMWaitNs)) {
      atomicOr(a.status, 2u);
      abort_flag = 1;
    } else if (tid == 0) {
      --pending;
    }
    // ---- the unit's tables: entry (row pair kq, rank r) per thread
    {
      const int h = u % H;
      const float d = reinterpret_cast<const float*>(stg + L.dt)[u & 3];
      const float lm = reinterpret_cast<const float*>(stg + L.lm)[u & 3];
      const float alpha = expf(d * sA[h]);
      const float gamma = lm * d, bhat = (1.f - lm) * d;
      const __nv_bfloat16* sB = reinterpret_cast<const __nv_bfloat16*>(stg + L.B);
      const __nv_bfloat16* sBp =
          has_prev ? reinterpret_cast<const __nv_bfloat16*>(stg + L.Bp) : nullptr;
      const __nv_bfloat16* sC = reinterpret_cast<const __nv_bfloat16*>(stg + L.C);
      const float* sbb = a.B_bias ? reinterpret_cast<const float*>(stg + L.bb) : nullptr;
      const float* scb = a.C_bias ? reinterpret_cast<const float*>(stg + L.cb) : nullptr;
      const float* sth = reinterpret_cast<const float*>(stg + L.th);
      for (int e = tid; e < K2 * kMR; e += kMThreads) {
        const int kq = e / kMR, r = e - kq * kMR;
        table_entry(T, kq, r, alpha, gamma, bhat, d * sth[kq], sB, sBp, sC, sbb, scb);
      }
    }
    // this warp's state columns and X fragment into registers, so that the
    // stage is free after the barrier
    float2 h0[NT], h1[NT];
    load_state<NT>(h0, h1, stg, L.half, g, p0);
    const uint32_t bx = x_fragment(stg + L.x, has_prev ? stg + L.xp : nullptr, warp, g, tq);
    __syncthreads();
    if (*reinterpret_cast<volatile int*>(&abort_flag)) break;  // uniform: read after the barrier
    // every warp is done with this stage: refill it two units ahead
    if (tid == 0) {
      const int un = u + kMStages * (int)gridDim.x;
      if (un < units) {
        issue(un, s);
        ++pending;
      }
    }
    token_step<NT, true>(h0, h1, T, bx, a.state + (int64_t)u * N * kMP,
                         static_cast<__nv_bfloat16*>(a.out) + ((int64_t)u * kMP + 8 * warp) * kMR,
                         g, tq, p0);
  }
  // after an early exit, let the copies in flight land before the CTA ends
  __syncthreads();
  if (tid == 0 && pending > 0) {
    for (int j = 0; j < kMStages; ++j, ++k) {
      const int u = blockIdx.x + k * (int)gridDim.x;
      if (u >= units) break;
      ptx::mbar_wait(&full[k % kMStages], (uint32_t)((k / kMStages) & 1), kMWaitNs);
    }
  }
}

// ------------------------------------------------------------- K tokens

// Shared memory of the K-token kernel: region S (the state, then the tables of
// a window of W tokens), then the block's activations: per token x [P][R],
// B and C [N][R] (bf16), theta [N/2]; x_prev, B_prev; the biases; dt, lambda [K].
struct TokMmaLayout {
  uint32_t half, tab, W;
  uint32_t X, Bm, Cm, TH, XP, BP, BB, CB, DT, LM;
  uint32_t copy_bytes, bytes;
};

inline TokMmaLayout tok_mma_layout(const TokensArgs& a) {
  const uint64_t N = a.N, P = kMP, R = kMR, K = a.K;
  const bool prev = a.B_prev != nullptr;
  TokMmaLayout L{};
  L.half = (uint32_t)(N * 32 * 4);
  L.tab = mma_table_bytes(N);
  uint32_t o = 0;
  L.X = o; o += (uint32_t)(K * P * R * 2);
  L.Bm = o; o += (uint32_t)(K * N * R * 2);
  L.Cm = o; o += (uint32_t)(K * N * R * 2);
  L.TH = o; o += (uint32_t)(K * N / 2 * 4);
  L.XP = o; o += prev ? (uint32_t)(P * R * 2) : 0u;
  L.BP = o; o += prev ? (uint32_t)(N * R * 2) : 0u;
  L.BB = o; o += a.B_bias ? (uint32_t)(N * R * 4) : 0u;
  L.CB = o; o += a.C_bias ? (uint32_t)(N * R * 4) : 0u;
  L.copy_bytes = o;
  L.DT = o; o += up16m(K * 4);
  L.LM = o; o += up16m(K * 4);
  const uint64_t acts = o;
  // region S takes what is left of the budget, at least the state
  const uint64_t avail = kMSmemMax > 1024 + acts ? kMSmemMax - 1024 - acts : 0;
  uint64_t W = avail / L.tab;
  if (W > K) W = K;
  L.W = (uint32_t)W;
  const uint64_t S = up1k(W * L.tab > 2ull * L.half ? W * L.tab : 2ull * L.half);
  L.X += (uint32_t)S; L.Bm += (uint32_t)S; L.Cm += (uint32_t)S; L.TH += (uint32_t)S;
  L.XP += (uint32_t)S; L.BP += (uint32_t)S; L.BB += (uint32_t)S; L.CB += (uint32_t)S;
  L.DT += (uint32_t)S; L.LM += (uint32_t)S;
  L.bytes = (uint32_t)(1024 + S + acts);
  return L;
}

template <int NT>
__global__ void __launch_bounds__(kMThreads, 2)
    decode_tokens_mma_kernel(const __grid_constant__ CUtensorMap tm_state, TokensArgs a,
                             TokMmaLayout L) {
  extern __shared__ __align__(16) uint8_t dsm_raw[];
  uint8_t* dsm = dsm_raw + ((1024u - (ptx::smem_addr(dsm_raw) & 1023u)) & 1023u);
  __shared__ uint64_t full;
  __shared__ int abort_flag;
  const int N = (int)a.N, K2 = N / 2, K = (int)a.K, H = (int)a.H;
  const int u = blockIdx.x, b = u / H, h = u - b * H, gi = h / (int)(a.H / a.G);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int p0 = 8 * warp + 2 * tq;
  const bool has_prev = a.B_prev != nullptr;
  const int64_t nr = (int64_t)N * kMR, pr = (int64_t)kMP * kMR;

  if (tid == 0) {
    abort_flag = 0;
    ptx::mbar_init(&full, 1);
    ptx::fence_mbar_init();
    uint64_t* bar = &full;
    ptx::mbar_arrive_expect_tx(bar, 2 * L.half + L.copy_bytes);
    tma_state(dsm, L.half, &tm_state, bar, u);
    const __nv_bfloat16* X = static_cast<const __nv_bfloat16*>(a.x);
    const __nv_bfloat16* Bg = static_cast<const __nv_bfloat16*>(a.B);
    const __nv_bfloat16* Cg = static_cast<const __nv_bfloat16*>(a.C);
    for (int t = 0; t < K; ++t) {
      const int64_t bt = (int64_t)b * K + t;
      ptx::bulk_load(dsm + L.X + t * pr * 2, X + (bt * H + h) * pr, (uint32_t)(pr * 2), bar);
      ptx::bulk_load(dsm + L.Bm + t * nr * 2, Bg + (bt * a.G + gi) * nr, (uint32_t)(nr * 2), bar);
      ptx::bulk_load(dsm + L.Cm + t * nr * 2, Cg + (bt * a.G + gi) * nr, (uint32_t)(nr * 2), bar);
      ptx::bulk_load(dsm + L.TH + t * K2 * 4, a.theta + (bt * a.G + gi) * K2, (uint32_t)K2 * 4, bar);
    }
    if (has_prev) {
      ptx::bulk_load(dsm + L.XP, static_cast<const __nv_bfloat16*>(a.x_prev) + (int64_t)u * pr,
                     (uint32_t)(pr * 2), bar);
      ptx::bulk_load(dsm + L.BP,
                     static_cast<const __nv_bfloat16*>(a.B_prev) + ((int64_t)b * a.G + gi) * nr,
                     (uint32_t)(nr * 2), bar);
    }
    if (a.B_bias) ptx::bulk_load(dsm + L.BB, a.B_bias + (int64_t)h * nr, (uint32_t)nr * 4, bar);
    if (a.C_bias) ptx::bulk_load(dsm + L.CB, a.C_bias + (int64_t)h * nr, (uint32_t)nr * 4, bar);
  }
  float* sdt = reinterpret_cast<float*>(dsm + L.DT);
  float* slm = reinterpret_cast<float*>(dsm + L.LM);
  for (int t = tid; t < K; t += kMThreads) {
    const int64_t i = ((int64_t)b * K + t) * H + h;
    sdt[t] = a.dt[i];
    slm[t] = a.lam[i];
  }
  const float A_h = a.A[h];
  __syncthreads();  // the barrier's initialisation and dt, lambda are visible
  if (!ptx::mbar_wait(&full, 0u, kMWaitNs)) {
    atomicOr(a.status, 2u);
    abort_flag = 1;
  }
  float2 h0[NT], h1[NT];
  load_state<NT>(h0, h1, dsm, L.half, g, p0);
  __syncthreads();
  if (*reinterpret_cast<volatile int*>(&abort_flag)) {
    // let the copies in flight land before the CTA ends; the state stays as it was
    if (tid == 0) ptx::mbar_wait(&full, 0u, kMWaitNs);
    return;
  }

  const __nv_bfloat16* sB = reinterpret_cast<const __nv_bfloat16*>(dsm + L.Bm);
  const __nv_bfloat16* sC = reinterpret_cast<const __nv_bfloat16*>(dsm + L.Cm);
  const float* sth = reinterpret_cast<const float*>(dsm + L.TH);
  const float* sbb = a.B_bias ? reinterpret_cast<const float*>(dsm + L.BB) : nullptr;
  const float* scb = a.C_bias ? reinterpret_cast<const float*>(dsm + L.CB) : nullptr;
  const __nv_bfloat16* sBP = has_prev ? reinterpret_cast<const __nv_bfloat16*>(dsm + L.BP) : nullptr;
  const int W = (int)L.W;
  for (int w0 = 0; w0 < K; w0 += W) {
    const int nw = K - w0 < W ? K - w0 : W;
    // tables of tokens w0 .. w0 + nw - 1 (region S: the state's copy is in registers)
    for (int e = tid; e < nw * K2 * kMR; e += kMThreads) {
      const int j = e / (K2 * kMR), rem = e - j * (K2 * kMR);
      const int kq = rem / kMR, r = rem - kq * kMR, t = w0 + j;
      const float d = sdt[t], lm = slm[t];
      const __nv_bfloat16* bp = t > 0 ? sB + (int64_t)(t - 1) * nr : sBP;
      table_entry(tok_tab(dsm + (size_t)j * L.tab, N), kq, r, expf(d * A_h), lm * d,
                  (1.f - lm) * d, d * sth[t * K2 + kq], sB + (int64_t)t * nr, bp,
                  sC + (int64_t)t * nr, sbb, scb);
    }
    __syncthreads();
    for (int j = 0; j < nw; ++j) {
      const int t = w0 + j;
      const uint8_t* xt = dsm + L.X + (size_t)t * pr * 2;
      const uint8_t* xpt = t > 0 ? xt - pr * 2 : (has_prev ? dsm + L.XP : nullptr);
      const uint32_t bx = x_fragment(xt, xpt, warp, g, tq);
      __nv_bfloat16* yw = static_cast<__nv_bfloat16*>(a.out) +
                          ((((int64_t)b * K + t) * H + h) * kMP + 8 * warp) * kMR;
      token_step<NT, false>(h0, h1, tok_tab(dsm + (size_t)j * L.tab, N), bx, nullptr, yw, g, tq,
                            p0);
    }
    if (w0 + nw < K) __syncthreads();  // the next window's tables overwrite these
  }
  float* gst = a.state + (int64_t)u * N * kMP;
#pragma unroll
  for (int rt = 0; rt < NT; ++rt) {
    const int n0 = 2 * (8 * rt + g);
    *reinterpret_cast<float2*>(gst + (int64_t)n0 * kMP + p0) = h0[rt];
    *reinterpret_cast<float2*>(gst + (int64_t)(n0 + 1) * kMP + p0) = h1[rt];
  }
}

// ------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFnM)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The state [units][N][64] fp32 as a 3-D tensor {64, N, units}: boxes of 32
// columns x N rows, 128-byte swizzled.
bool make_state_map(CUtensorMap* m, float* state, int64_t units, int64_t N) {
  static EncodeTiledFnM fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<EncodeTiledFnM>(ptr);
  }
  cuuint64_t dims[3] = {(cuuint64_t)kMP, (cuuint64_t)N, (cuuint64_t)units};
  cuuint64_t strides[2] = {(cuuint64_t)kMP * 4, (cuuint64_t)N * kMP * 4};
  cuuint32_t box[3] = {32, (cuuint32_t)N, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, state, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 148;
  return sms;
}

template <int NT>
cudaError_t launch_one(const CUtensorMap& tm, const DecodeArgs& a, const MmaLayout& L, size_t smem,
                       int grid, int units, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<NT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode_mma_kernel<NT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           100);
  if (e != cudaSuccess) return e;
  decode_mma_kernel<NT><<<grid, kMThreads, smem, s>>>(tm, a, L, units);
  return cudaGetLastError();
}

template <int NT>
cudaError_t launch_tok(const CUtensorMap& tm, const TokensArgs& a, const TokMmaLayout& L,
                       cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(decode_tokens_mma_kernel<NT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.bytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode_tokens_mma_kernel<NT>,
                           cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  decode_tokens_mma_kernel<NT><<<(unsigned)(a.batch * a.H), kMThreads, L.bytes, s>>>(tm, a, L);
  return cudaGetLastError();
}

}  // namespace

bool decode_mma_ok(const DecodeArgs& a, bool bf16) {
  if (!bf16 || a.R != kMR || a.P != kMP || a.status == nullptr) return false;
  if (a.N < 16 || a.N > 16 * kMaxNT || a.N % 16 != 0) return false;
  if ((a.batch * a.H) % 4 != 0 || a.batch * a.H > 0x7fffffffLL) return false;
  const void* ptrs[] = {a.state, a.x, a.x_prev, a.B, a.B_prev, a.C, a.theta,
                        a.B_bias, a.C_bias, a.dt, a.lam, a.out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return false;
  const MmaLayout L = mma_layout(a);
  return mma_smem_bytes(a, L) <= kMSmemMax;
}

cudaError_t launch_decode_mma(const DecodeArgs& a, cudaStream_t s) {
  CUtensorMap tm;
  if (!make_state_map(&tm, a.state, a.batch * a.H, a.N)) return cudaErrorInvalidValue;
  const MmaLayout L = mma_layout(a);
  const size_t smem = mma_smem_bytes(a, L);
  const int units = (int)(a.batch * a.H);
  const int sms = sm_count();
  const int grid = units < 2 * sms ? units : 2 * sms;
  switch (a.N / 16) {
    case 1: return launch_one<1>(tm, a, L, smem, grid, units, s);
    case 2: return launch_one<2>(tm, a, L, smem, grid, units, s);
    case 3: return launch_one<3>(tm, a, L, smem, grid, units, s);
    case 4: return launch_one<4>(tm, a, L, smem, grid, units, s);
    case 5: return launch_one<5>(tm, a, L, smem, grid, units, s);
    case 6: return launch_one<6>(tm, a, L, smem, grid, units, s);
    case 7: return launch_one<7>(tm, a, L, smem, grid, units, s);
    case 8: return launch_one<8>(tm, a, L, smem, grid, units, s);
    default: return cudaErrorInvalidValue;
  }
}

bool tokens_mma_ok(const TokensArgs& a, bool bf16) {
  if (!bf16 || a.R != kMR || a.P != kMP || a.status == nullptr) return false;
  if (a.N < 16 || a.N > 16 * kMaxNT || a.N % 16 != 0) return false;
  if (a.K < 1 || a.batch * a.H < 1 || a.batch * a.H > 0x7fffffffLL) return false;
  const void* ptrs[] = {a.state, a.x, a.x_prev, a.B, a.B_prev, a.C, a.theta, a.B_bias, a.C_bias,
                        a.out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return false;
  const TokMmaLayout L = tok_mma_layout(a);
  return L.W >= 1 && L.bytes <= kMSmemMax;
}

cudaError_t launch_tokens_mma(const TokensArgs& a, cudaStream_t s) {
  CUtensorMap tm;
  if (!make_state_map(&tm, a.state, a.batch * a.H, a.N)) return cudaErrorInvalidValue;
  const TokMmaLayout L = tok_mma_layout(a);
  switch (a.N / 16) {
    case 1: return launch_tok<1>(tm, a, L, s);
    case 2: return launch_tok<2>(tm, a, L, s);
    case 3: return launch_tok<3>(tm, a, L, s);
    case 4: return launch_tok<4>(tm, a, L, s);
    case 5: return launch_tok<5>(tm, a, L, s);
    case 6: return launch_tok<6>(tm, a, L, s);
    case 7: return launch_tok<7>(tm, a, L, s);
    case 8: return launch_tok<8>(tm, a, L, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace m3
