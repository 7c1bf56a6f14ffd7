// One decode token of the Mamba-3 scan at MIMO rank R = 4 (bf16 activations,
// P = 64), with the rank-R update on the tensor cores.
//
// For every (batch, head) the step is (Prop. 1 and the rotation, sec. 4.1 and
// 4.2 of "MAMBA-3: IMPROVED SEQUENCE MODELING USING STATE SPACE PRINCIPLES"
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
// 8w .. 8w + 7 over all rows, so its partial y needs only a reduction across
// its own lanes.
//
// The step is bound by HBM traffic (the fp32 state is read and written once).
// A persistent kernel (two 256-thread CTAs per SM) streams the (b, h) units
// through two stages of shared memory: the state by TMA with the 128-byte
// swizzle (so that the MMA layout's 8 rows x 8 columns loads are free of bank
// conflicts), the token's activations by bulk copies. Every wait is bounded;
// an expired wait sets the status word and the CTA leaves at the next barrier.
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

__host__ __device__ constexpr uint32_t up16m(uint64_t v) { return (uint32_t)((v + 15) & ~15ull); }
__host__ __device__ constexpr uint32_t up1k(uint64_t v) { return (uint32_t)((v + 1023) & ~1023ull); }

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

// Per-unit tables (two sets, alternating units): U high and low parts
// [N/2 pairs][kPairWords] (row 2k at words 0-3, row 2k + 1 at words 4-7, each
// as 2R = 8 bf16), C + bias [N][R] fp32, alpha (cos, sin) [N/2].
__host__ __device__ inline uint32_t mma_table_bytes(int64_t N) {
  return (uint32_t)(2 * (N / 2) * kPairWords * 4 + N * kMR * 4 + (N / 2) * 8);
}

inline size_t mma_smem_bytes(const DecodeArgs& a, const MmaLayout& L) {
  return 1024 + (size_t)kMStages * L.bytes + 2 * (size_t)mma_table_bytes(a.N) + 4 * (size_t)a.H;
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

// Byte offset of state element (n, col) in a stage: column half, row n (128
// bytes), 16-byte chunk XOR the row's low three bits (the TMA 128B swizzle).
__device__ __forceinline__ uint32_t st_off(uint32_t half_bytes, uint32_t n, uint32_t col) {
  const uint32_t cl = col & 31u;
  return (col >> 5) * half_bytes + n * 128u + ((((cl >> 2) ^ n) & 7u) << 4) + (cl & 3u) * 4u;
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
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(ptx::smem_addr(st)),
        "l"(reinterpret_cast<uint64_t>(&tm_state)), "r"(ptx::smem_addr(bar)), "r"(0), "r"(0), "r"(u)
        : "memory");
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(ptx::smem_addr(st + L.half)),
        "l"(reinterpret_cast<uint64_t>(&tm_state)), "r"(ptx::smem_addr(bar)), "r"(32), "r"(0), "r"(u)
        : "memory");
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
    uint8_t* tab = tables + (size_t)(k & 1) * tbytes;
    uint32_t* Uh = reinterpret_cast<uint32_t*>(tab);
    uint32_t* Ul = Uh + K2 * kPairWords;
    float* cd = reinterpret_cast<float*>(Ul + K2 * kPairWords);  // C + bias [N][R]
    float2* rd = reinterpret_cast<float2*>(cd + N * kMR);         // alpha (cos, sin) [K2]
    if (!ptx::mbar_wait(&full[s], (uint32_t)((k / kMStages) & 1), kMWaitNs)) {
      atomicOr(a.status, 2u);
      abort_flag = 1;
    } else if (tid == 0) {
      --pending;
    }
    // ---- per-unit tables: entry (row pair kq, rank r) per thread
    const int h = u % H;
    const float d = reinterpret_cast<const float*>(stg + L.dt)[u & 3];
    const float lm = reinterpret_cast<const float*>(stg + L.lm)[u & 3];
    const float alpha = expf(d * sA[h]);
    const float gamma = lm * d, bhat = (1.f - lm) * d;
    {
      const __nv_bfloat16* sB = reinterpret_cast<const __nv_bfloat16*>(stg + L.B);
      const __nv_bfloat16* sBp = reinterpret_cast<const __nv_bfloat16*>(stg + L.Bp);
      const __nv_bfloat16* sC = reinterpret_cast<const __nv_bfloat16*>(stg + L.C);
      const float* sbb = reinterpret_cast<const float*>(stg + L.bb);
      const float* scb = reinterpret_cast<const float*>(stg + L.cb);
      const float* sth = reinterpret_cast<const float*>(stg + L.th);
      __nv_bfloat16* Uh16 = reinterpret_cast<__nv_bfloat16*>(Uh);
      __nv_bfloat16* Ul16 = reinterpret_cast<__nv_bfloat16*>(Ul);
      for (int e = tid; e < K2 * kMR; e += kMThreads) {
        const int kq = e / kMR, r = e - kq * kMR;
        float sn, cs;
        __sincosf(wrap_angle(d * sth[kq]), &sn, &cs);
        const float ac = alpha * cs, as = alpha * sn;
        const int i0 = 2 * kq * kMR + r, i1 = i0 + kMR;  // (row 2kq, r), (row 2kq + 1, r)
        const float bb0 = a.B_bias ? sbb[i0] : 0.f, bb1 = a.B_bias ? sbb[i1] : 0.f;
        const float cb0 = a.C_bias ? scb[i0] : 0.f, cb1 = a.C_bias ? scb[i1] : 0.f;
        float u0 = 0.f, u1 = 0.f;
        if (has_prev) {
          const float q0 = bhat * (ld_act(sBp + i0) + bb0), q1 = bhat * (ld_act(sBp + i1) + bb1);
          u0 = fmaf(ac, q0, -as * q1);
          u1 = fmaf(as, q0, ac * q1);
        }
        const float g0 = gamma * (ld_act(sB + i0) + bb0), g1 = gamma * (ld_act(sB + i1) + bb1);
        // U row 2kq: [u0 | g0] at bf16 index r and R + r; row 2kq + 1 eight further
        const float v[4] = {u0, g0, u1, g1};
        const int idx[4] = {r, kMR + r, 2 * kMR + r, 3 * kMR + r};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const __nv_bfloat16 hi = __float2bfloat16_rn(v[q]);
          Uh16[kq * 2 * kPairWords + idx[q]] = hi;
          Ul16[kq * 2 * kPairWords + idx[q]] = __float2bfloat16_rn(v[q] - __bfloat162float(hi));
        }
        cd[i0] = ld_act(sC + i0) + cb0;
        cd[i1] = ld_act(sC + i1) + cb1;
        if (r == 0) rd[kq] = make_float2(ac, as);
      }
    }
    // this warp's state columns p0, p0 + 1 of every row pair, and its X
    // fragment, into registers, so that the stage is free after the barrier
    const int p0 = 8 * warp + 2 * tq;
    float2 h0[NT], h1[NT];  // rows 2kq and 2kq + 1, kq = 8 rt + g
    {
      // row 2kq = 2g + 16 rt: the swizzle phase (row & 7) is the same for every rt
      const uint8_t* r0 = stg + st_off(L.half, 2u * g, (uint32_t)p0);
      const uint8_t* r1 = stg + st_off(L.half, 2u * g + 1u, (uint32_t)p0);
#pragma unroll
      for (int rt = 0; rt < NT; ++rt) {
        h0[rt] = *reinterpret_cast<const float2*>(r0 + rt * 16 * 128);
        h1[rt] = *reinterpret_cast<const float2*>(r1 + rt * 16 * 128);
      }
    }
    // X fragment: X[p = 8 warp + g][k = 2 tq, 2 tq + 1]; k < R is x_prev, else x
    uint32_t bx;
    {
      const int pcol = 8 * warp + g;
      const uint32_t* src = reinterpret_cast<const uint32_t*>(stg + (tq < 2 ? L.xp : L.x));
      bx = (tq < 2 && !has_prev) ? 0u : src[pcol * (kMR / 2) + (tq & 1)];
    }
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

    // ---- h' = alpha Rot h + U X^T over the warp's 8 columns, y += C^T h'
    float2 yv[kMR];  // (y[p0][r], y[p0 + 1][r])
#pragma unroll
    for (int r = 0; r < kMR; ++r) yv[r] = make_float2(0.f, 0.f);
    float* gst = a.state + (int64_t)u * N * kMP;
#pragma unroll
    for (int rt = 0; rt < NT; ++rt) {
      const int kq = 8 * rt + g;  // this thread's row pair
      float dacc[4] = {0.f, 0.f, 0.f, 0.f};
      mma_bf16_16x8x8(dacc, Uh[kq * kPairWords + tq], Uh[kq * kPairWords + 4 + tq], bx);
      mma_bf16_16x8x8(dacc, Ul[kq * kPairWords + tq], Ul[kq * kPairWords + 4 + tq], bx);
      const uint32_t n0 = 2u * kq, n1 = n0 + 1u;
      const float2 h0v = h0[rt], h1v = h1[rt];
      const float2 rot = rd[kq];
      const float2 ac2 = make_float2(rot.x, rot.x), as2 = make_float2(rot.y, rot.y);
      const float2 nas2 = make_float2(-rot.y, -rot.y);
      // rows 2kq, 2kq + 1: alpha [[c, -s], [s, c]] (h0, h1) + U X^T
      const float2 r0 = ptx::fma2(ac2, h0v, ptx::fma2(nas2, h1v, make_float2(dacc[0], dacc[1])));
      const float2 r1 = ptx::fma2(as2, h0v, ptx::fma2(ac2, h1v, make_float2(dacc[2], dacc[3])));
      *reinterpret_cast<float2*>(gst + (int64_t)n0 * kMP + p0) = r0;
      *reinterpret_cast<float2*>(gst + (int64_t)n1 * kMP + p0) = r1;
      const float4 ce = *reinterpret_cast<const float4*>(cd + n0 * kMR);
      const float4 co = *reinterpret_cast<const float4*>(cd + n1 * kMR);
      const float cev[4] = {ce.x, ce.y, ce.z, ce.w}, cov[4] = {co.x, co.y, co.z, co.w};
#pragma unroll
      for (int r = 0; r < kMR; ++r)
        yv[r] = ptx::fma2(make_float2(cev[r], cev[r]), r0,
                          ptx::fma2(make_float2(cov[r], cov[r]), r1, yv[r]));
    }
    // sum the eight values v[4c + r] = y[p0 + c][r] over the warp's row pairs
    // (the lanes that differ in g), halving the values at each step so that
    // lane (g, tq) ends with v[g] in full
    float w[4], z[2], t;
    {
      const bool b2 = (g & 4) != 0, b1 = (g & 2) != 0, b0 = (g & 1) != 0;
      float v[8];
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
      t = (b0 ? z[1] : z[0]) + __shfl_xor_sync(0xffffffffu, b0 ? z[0] : z[1], 4);
    }
    // v[g] is y[p0 + (g >> 2)][g & 3], at offset 8 tq + g of the warp's 32
    // outputs; even g stores itself and its odd neighbour as one bf16 pair
    const float t_next = __shfl_xor_sync(0xffffffffu, t, 4);
    if ((g & 1) == 0) {
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + ((int64_t)u * kMP + 8 * warp) * kMR;
      *reinterpret_cast<uint32_t*>(out + 8 * tq + g) = bf16_pair(t, t_next);
    }
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

typedef CUresult (*EncodeTiledFnM)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The state [b H][N][64] fp32 as a 3-D tensor {64, N, b H}: boxes of 32 columns
// x N rows, 128-byte swizzled.
bool make_state_map(CUtensorMap* m, const DecodeArgs& a) {
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
  const uint64_t units = (uint64_t)(a.batch * a.H);
  cuuint64_t dims[3] = {(cuuint64_t)kMP, (cuuint64_t)a.N, (cuuint64_t)units};
  cuuint64_t strides[2] = {(cuuint64_t)kMP * 4, (cuuint64_t)a.N * kMP * 4};
  cuuint32_t box[3] = {32, (cuuint32_t)a.N, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.state, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool decode_mma_ok(const DecodeArgs& a, bool bf16) {
  auto al = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!bf16 || a.R != kMR || a.P != kMP || a.status == nullptr) return false;
  if (a.N < 16 || a.N > 16 * kMaxNT || a.N % 16 != 0) return false;
  if ((a.batch * a.H) % 4 != 0 || a.batch * a.H > 0x7fffffffLL) return false;
  if (!al(a.state) || !al(a.x) || !al(a.x_prev) || !al(a.B) || !al(a.B_prev) || !al(a.C) ||
      !al(a.theta) || !al(a.B_bias) || !al(a.C_bias) || !al(a.dt) || !al(a.lam) || !al(a.out))
    return false;
  const MmaLayout L = mma_layout(a);
  return mma_smem_bytes(a, L) <= 112 * 1024;
}

template <int NT>
cudaError_t launch_nt(const CUtensorMap& tm, const DecodeArgs& a, const MmaLayout& L, size_t smem,
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

cudaError_t launch_decode_mma(const DecodeArgs& a, cudaStream_t s) {
  CUtensorMap tm;
  if (!make_state_map(&tm, a)) return cudaErrorInvalidValue;
  const MmaLayout L = mma_layout(a);
  const size_t smem = mma_smem_bytes(a, L);
  int dev = 0, sms = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const int units = (int)(a.batch * a.H);
  const int grid = units < 2 * sms ? units : 2 * sms;
  switch (a.N / 16) {
    case 1: return launch_nt<1>(tm, a, L, smem, grid, units, s);
    case 2: return launch_nt<2>(tm, a, L, smem, grid, units, s);
    case 3: return launch_nt<3>(tm, a, L, smem, grid, units, s);
    case 4: return launch_nt<4>(tm, a, L, smem, grid, units, s);
    case 5: return launch_nt<5>(tm, a, L, smem, grid, units, s);
    case 6: return launch_nt<6>(tm, a, L, smem, grid, units, s);
    case 7: return launch_nt<7>(tm, a, L, smem, grid, units, s);
    case 8: return launch_nt<8>(tm, a, L, smem, grid, units, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace m3
