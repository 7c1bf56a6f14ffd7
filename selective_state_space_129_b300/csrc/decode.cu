// One decode token of the Mamba-3 scan, state streamed once.
//
// For every (batch, head):
//   G   = h + beta_hat (B_prev + bias) x_prev^T
//   h' = alpha Rot(Delta theta) G + gamma (B + bias) x^T
//   y   = (C + bias)^T h'                                   (P x R, stored [P][R])
// which is the recurrence of Prop. 1 with the state rotation of the
// complex-valued SSM (sec. 4.1 and 4.2 of the page
// "MAMBA-3: IMPROVED SEQUENCE MODELING USING STATE SPACE PRINCIPLES" (aipaper.cc); the
// rotation matrix of sec. 2.2 of
// "State Space Models 家族对比分析：S4 → Mamba → Mamba-2 → Mamba-3" (metaphor-xennon blog)),
// with MIMO rank R (sec. 3 of "Mamba-3: Improved Sequence Modeling using State Space Principles" (papernotes.org)).
//
// The step is bound by HBM traffic: the fp32 state (N x P per head) is read
// and written once, everything else is a few KB per head. The rank-R
// products are formed on the CUDA cores in registers while the state streams
// (about 3R + 2 FMAs per state element); the rank-4 step is the one where this
// arithmetic and the per-(b, h) set-up start to show next to the stream.
//
// Two kernels. The streaming kernel (further below) is used whenever its
// copy-engine alignment rules hold. The one-CTA-per-(batch, head) kernel here
// takes every other shape: 256 threads; a work item is one rotating row pair
// (2k, 2k+1) times four consecutive columns, loaded as two 16-byte vectors, so
// that a warp reads 2 x 256 contiguous bytes per instruction. Each thread
// keeps a fixed column quad, so its x / x_prev values and its partial y stay
// in registers. The first items' state loads are issued before the per-head
// coefficients are prepared, so that they are in flight during that set-up;
// the partial y are reduced with warp shuffles and one shared-memory pass,
// without atomics.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

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


// ---------------------------------------------------------------- streaming
// Persistent form of the same step. A CTA walks the (batch, head) units
// u = blockIdx.x, + gridDim.x, ...; its thread 0 stages each unit's state and
// activations into shared memory with bulk asynchronous copies, kStages units
// ahead, so that the state stream from HBM does not wait for the arithmetic or
// for the per-unit barriers. The new state goes straight from registers to
// global memory. Used when every per-unit block is 16-byte aligned and a
// multiple of 16 bytes long (the copy engine's rule); other shapes take the
// kernel above.
constexpr int kSThreads = 256;
constexpr int kSWarps = kSThreads / 32;
constexpr int kStages = 2;
constexpr uint64_t kStreamWaitNs = 2000000000ull;  // 2 s per wait

__host__ __device__ inline uint32_t up16(uint64_t v) { return (uint32_t)((v + 15) & ~uint64_t(15)); }

// Byte offsets of one unit's blocks inside a stage.
struct StreamLayout {
  uint32_t st, x, xp, B, Bp, C, th, bb, cb, dt, lm, bytes, tx;
};

inline StreamLayout stream_layout(const DecodeArgs& a, int act) {
  const uint64_t N = a.N, P = a.P, R = a.R;
  const bool prev = a.B_prev != nullptr;
  StreamLayout L{};
  uint32_t o = 0;
  L.st = o; o += up16(N * P * 4);
  L.x = o; o += up16(P * R * act);
  L.xp = o; o += prev ? up16(P * R * act) : 0u;
  L.B = o; o += up16(N * R * act);
  L.Bp = o; o += prev ? up16(N * R * act) : 0u;
  L.C = o; o += up16(N * R * act);
  L.th = o; o += up16(N / 2 * 4);
  L.bb = o; o += a.B_bias ? up16(N * R * 4) : 0u;
  L.cb = o; o += a.C_bias ? up16(N * R * 4) : 0u;
  L.dt = o; o += 16;
  L.lm = o; o += 16;
  L.bytes = o;
  L.tx = o;  // every block is copied whole (sizes are multiples of 16)
  return L;
}

// Per-unit coefficient tables: 3NR + N floats. R = 1: gamma (B + bias),
// beta_hat (B_prev + bias), C + bias as [N][R] rows and alpha cos, alpha sin
// as [N/2]. R > 1: the rotation is folded into the B_prev term (see the
// kernel): U [N][2R] rows, C + bias [N][R] rows, (alpha cos, alpha sin) [N/2].
__host__ __device__ inline size_t stream_coef_floats(size_t N, size_t R) { return 3 * N * R + N; }
// Whether each warp prepares the coefficient rows of its own row pairs (no
// block-wide barrier between preparation and items) or the whole CTA prepares
// every row and meets at a barrier.
__host__ __device__ constexpr bool stream_warp_prep(int R) { return R == 1; }
// Two partial-y tables with per-warp preparation (no block-wide barrier
// between one unit's final sum and the next unit's items), else one.
__host__ __device__ inline int stream_yred_tables(int R) { return stream_warp_prep(R) ? 2 : 1; }

// Partial y of warp w, column 4q + c, rank r at yred[(w 4R + c R + r)(P/4 + 1) + q]:
// the lanes of a warp (consecutive q) store to consecutive words, and the
// padding keeps the reads of the final sum (consecutive (p, r)) off shared banks.
inline size_t stream_smem_bytes(const DecodeArgs& a, const StreamLayout& L) {
  const size_t N = a.N, P = a.P, R = a.R;
  return (size_t)kStages * L.bytes +
         sizeof(float) * (stream_coef_floats(N, R) +
                          stream_yred_tables(a.R) * (size_t)kSWarps * R * (P + 4) + (size_t)a.H);
}

// The 4 x R activations of one column quad (4 R consecutive elements of a
// 16-byte aligned block, at an offset that is a multiple of 8 bytes) with
// vector loads.
template <typename T, int R>
__device__ __forceinline__ void ld_quad(const T* p, float (&v)[4][R]) {
  constexpr int kBytes = 4 * R * (int)sizeof(T);
  if constexpr (sizeof(T) == 2) {
    uint32_t w[kBytes / 4];
    if constexpr (kBytes == 8) {
      const uint2 a = *reinterpret_cast<const uint2*>(p);
      w[0] = a.x; w[1] = a.y;
    } else {
#pragma unroll
      for (int k = 0; k < kBytes / 16; ++k) {
        const uint4 a = reinterpret_cast<const uint4*>(p)[k];
        w[4 * k] = a.x; w[4 * k + 1] = a.y; w[4 * k + 2] = a.z; w[4 * k + 3] = a.w;
      }
    }
#pragma unroll
    for (int i = 0; i < 4 * R; ++i)
      v[i / R][i % R] = __uint_as_float((i & 1) ? (w[i >> 1] & 0xffff0000u) : (w[i >> 1] << 16));
  } else {
#pragma unroll
    for (int k = 0; k < R; ++k) {
      const float4 a = reinterpret_cast<const float4*>(p)[k];
      const float e[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) v[(4 * k + j) / R][(4 * k + j) % R] = e[j];
    }
  }
}

template <typename T, int R>
__global__ void __launch_bounds__(kSThreads, 2)
    decode_stream_kernel(DecodeArgs a, StreamLayout L, int units) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ uint64_t full[kStages];
  __shared__ int abort_flag;
  const int N = (int)a.N, P = (int)a.P, K2 = N / 2, PQ = P / 4, H = (int)a.H;
  const int hpg = (int)(a.H / a.G);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float* coef = reinterpret_cast<float*>(dsm + (size_t)kStages * L.bytes);
  float* bg = coef;              // R = 1: gamma (B + bias)   [N][R]
  float* bp = bg + N * R;        //        beta_hat (B_prev + bias)  [N][R]
  float* cc = bp + N * R;        //        C + bias           [N][R]
  float* rc = cc + N * R;        //        alpha cos          [K2]
  float* rs = rc + K2;           //        alpha sin          [K2]
  float* ud = coef;              // R > 1: U                  [N][2R]
  float* cd = ud + 2 * N * R;    //        C + bias           [N][R]
  float* rd = cd + N * R;        //        alpha (cos, sin)   [K2][2]
  float* yred0 = coef + stream_coef_floats(N, R);  // partial y per warp (padded layout above)
  const int yred_floats = kSWarps * R * (P + 4);
  float* sA = yred0 + stream_yred_tables(R) * yred_floats;  // A [H]
  const bool has_prev = a.B_prev != nullptr;
  const int q = tid % PQ;  // this thread's column quad (PQ divides 32)
  const int items = K2 * PQ;

  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < kStages; ++s) ptx::mbar_init(&full[s], 1);
    ptx::fence_mbar_init();
  }
  for (int i = tid; i < H; i += kSThreads) sA[i] = a.A[i];
  __syncthreads();

  // thread 0: stage unit u into stage s
  auto issue = [&](int u, int s) {
    const int b = u / H, h = u - b * H, g = h / hpg;
    uint8_t* st = dsm + (size_t)s * L.bytes;
    uint64_t* bar = &full[s];
    const int64_t nr = (int64_t)N * R, pr = (int64_t)P * R;
    const int64_t bc = ((int64_t)b * a.G + g) * nr;
    ptx::fence_proxy_async_smem();  // earlier reads of the stage come first
    ptx::mbar_arrive_expect_tx(bar, L.tx);
    ptx::bulk_load(st + L.st, a.state + (int64_t)u * N * P, (uint32_t)N * P * 4, bar);
    ptx::bulk_load(st + L.x, static_cast<const T*>(a.x) + (int64_t)u * pr,
                   (uint32_t)(pr * sizeof(T)), bar);
    if (has_prev)
      ptx::bulk_load(st + L.xp, static_cast<const T*>(a.x_prev) + (int64_t)u * pr,
                     (uint32_t)(pr * sizeof(T)), bar);
    ptx::bulk_load(st + L.B, static_cast<const T*>(a.B) + bc, (uint32_t)(nr * sizeof(T)), bar);
    if (has_prev)
      ptx::bulk_load(st + L.Bp, static_cast<const T*>(a.B_prev) + bc, (uint32_t)(nr * sizeof(T)),
                     bar);
    ptx::bulk_load(st + L.C, static_cast<const T*>(a.C) + bc, (uint32_t)(nr * sizeof(T)), bar);
    ptx::bulk_load(st + L.th, a.theta + ((int64_t)b * a.G + g) * K2, (uint32_t)K2 * 4, bar);
    if (a.B_bias) ptx::bulk_load(st + L.bb, a.B_bias + (int64_t)h * nr, (uint32_t)nr * 4, bar);
    if (a.C_bias) ptx::bulk_load(st + L.cb, a.C_bias + (int64_t)h * nr, (uint32_t)nr * 4, bar);
    // dt, lambda of unit u: the aligned 16-byte window that holds them
    ptx::bulk_load(st + L.dt, a.dt + (u & ~3), 16u, bar);
    ptx::bulk_load(st + L.lm, a.lam + (u & ~3), 16u, bar);
  };
  if (tid == 0)
    for (int j = 0; j < kStages; ++j) {
      const int u = blockIdx.x + j * gridDim.x;
      if (u < units) issue(u, j);
    }

  int k = 0;
  for (int u = blockIdx.x; u < units; u += gridDim.x, ++k) {
    const int s = k % kStages;
    const uint8_t* stg = dsm + (size_t)s * L.bytes;
    // every lane waits for the stage; a warp whose wait ran out writes nothing
    const bool ok =
        __all_sync(0xffffffffu, ptx::mbar_wait(&full[s], (uint32_t)((k / kStages) & 1), kStreamWaitNs));
    if (!ok && lane == 0) {
      atomicOr(a.status, 2u);
      abort_flag = 1;
    }
    // At R = 1 each warp prepares the coefficient rows of the row pairs it
    // updates itself, so no block-wide barrier separates preparation and
    // items: its items are it = 32 warp + lane + j kSThreads, i.e. the 32 / PQ
    // row pairs from (32 warp + j kSThreads) / PQ for every j. At R > 1 the
    // CTA prepares all rows and meets at a barrier, which measured faster
    // (b128 H32 P64 N128 R4: 58 us per step against 65 us per-warp; R1: 45 us
    // per-warp against 47 us).
    constexpr bool kWarpPrep = stream_warp_prep(R);
    const int kpw = 32 / PQ;                                  // row pairs per block of 32 items
    const int nj = (items - 32 * warp + kSThreads - 1) / kSThreads;  // this warp's blocks
    const int h = u % H;
    const float d = reinterpret_cast<const float*>(stg + L.dt)[u & 3];
    const float lm = reinterpret_cast<const float*>(stg + L.lm)[u & 3];
    const float alpha = expf(d * sA[h]);
    const float gamma = lm * d, bhat = (1.f - lm) * d;
    const T* sB = reinterpret_cast<const T*>(stg + L.B);
    const T* sBp = reinterpret_cast<const T*>(stg + L.Bp);
    const T* sC = reinterpret_cast<const T*>(stg + L.C);
    const float* sbb = reinterpret_cast<const float*>(stg + L.bb);
    const float* scb = reinterpret_cast<const float*>(stg + L.cb);
    const float* sth = reinterpret_cast<const float*>(stg + L.th);
    // R > 1: the rotation is linear in the rows, so alpha Rot (beta_hat
    // (B_prev + bias) x_prev^T) = (alpha Rot beta_hat (B_prev + bias)) x_prev^T:
    // the rotated rows U[n][r] are formed once per unit, and the items apply
    // the rotation to the state alone. Entry (row pair kq, rank r):
    auto fold_prep = [&](int kq, int r) {
      float sn, cs;
      __sincosf(wrap_angle(d * sth[kq]), &sn, &cs);
      const float ac = alpha * cs, as = alpha * sn;
      const int i0 = 2 * kq * R + r, i1 = i0 + R;  // (row 2kq, r), (row 2kq + 1, r)
      const float bb0 = a.B_bias ? sbb[i0] : 0.f, bb1 = a.B_bias ? sbb[i1] : 0.f;
      const float cb0 = a.C_bias ? scb[i0] : 0.f, cb1 = a.C_bias ? scb[i1] : 0.f;
      float u0 = 0.f, u1 = 0.f;
      if (has_prev) {
        const float p0 = bhat * (ld_act(sBp + i0) + bb0), p1 = bhat * (ld_act(sBp + i1) + bb1);
        u0 = fmaf(ac, p0, -as * p1);
        u1 = fmaf(as, p0, ac * p1);
      }
      const float g0 = gamma * (ld_act(sB + i0) + bb0), g1 = gamma * (ld_act(sB + i1) + bb1);
      float* U0 = ud + 2 * kq * 2 * R;  // row 2kq: U[n][r] = rotated B_prev term, U[n][R + r] = B term
      U0[r] = u0;
      U0[R + r] = g0;
      U0[2 * R + r] = u1;  // row 2kq + 1
      U0[3 * R + r] = g1;
      cd[i0] = ld_act(sC + i0) + cb0;
      cd[i1] = ld_act(sC + i1) + cb1;
      if (r == 0) reinterpret_cast<float2*>(rd)[kq] = make_float2(ac, as);
    };
    if (!kWarpPrep) {
      for (int e = tid; ok && e < K2 * R; e += kSThreads) fold_prep(e / R, e % R);
      __syncthreads();
      if (abort_flag) break;  // uniform: read after the barrier
    } else if (R > 1 && ok && nj > 0) {
      for (int e = lane; e < nj * kpw * R; e += 32) {
        const int jj = e / (kpw * R), rem = e - jj * kpw * R;
        const int kq = (32 * warp + jj * kSThreads) / PQ + rem / R;
        if (kq < K2) fold_prep(kq, rem % R);
      }
    } else if (ok && nj > 0) {
      const int per_block = kpw * 2 * R;  // coefficient entries (row, rank) per block
      for (int e = lane; e < nj * per_block; e += 32) {
        const int jj = e / per_block, rem = e - jj * per_block;
        const int kq = (32 * warp + jj * kSThreads) / PQ + rem / (2 * R);
        if (kq >= K2) continue;  // past the last row pair (a partial block)
        const int i = 2 * kq * R + rem % (2 * R);  // index (n, r) of row n = 2 kq + (rem % 2R) / R
        const float bb = a.B_bias ? sbb[i] : 0.f;
        const float cb = a.C_bias ? scb[i] : 0.f;
        bg[i] = gamma * (ld_act(sB + i) + bb);
        bp[i] = has_prev ? bhat * (ld_act(sBp + i) + bb) : 0.f;
        cc[i] = ld_act(sC + i) + cb;
      }
      for (int e = lane; e < nj * kpw; e += 32) {
        const int jj = e / kpw;
        const int kq = (32 * warp + jj * kSThreads) / PQ + (e - jj * kpw);
        if (kq >= K2) continue;
        float sn, cs;
        __sincosf(wrap_angle(d * sth[kq]), &sn, &cs);
        rc[kq] = alpha * cs;
        rs[kq] = alpha * sn;
      }
    }
    __syncwarp();
    const T* sx = reinterpret_cast<const T*>(stg + L.x);
    const T* sxp = reinterpret_cast<const T*>(stg + L.xp);
    float xr[4][R], xpr[4][R], yp[4][R];
    ld_quad<T, R>(sx + 4 * q * R, xr);
    if (has_prev) {
      ld_quad<T, R>(sxp + 4 * q * R, xpr);
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int r = 0; r < R; ++r) xpr[c][r] = 0.f;
    }
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int r = 0; r < R; ++r) yp[c][r] = 0.f;

    const float* sst = reinterpret_cast<const float*>(stg + L.st);
    float* gst = a.state + (int64_t)u * N * P;
    // with per-warp preparation two tables alternate: the last unit's sum may still read the other
    float* yred = yred0 + (kWarpPrep ? (k & 1) * yred_floats : 0);
    if constexpr (R == 1) {
      for (int it = tid; ok && it < items; it += kSThreads) {
        const int kq = it / PQ;
        float4 h0 = *reinterpret_cast<const float4*>(sst + (2 * kq) * P + 4 * q);
        float4 h1 = *reinterpret_cast<const float4*>(sst + (2 * kq + 1) * P + 4 * q);
        const float bp0 = bp[2 * kq], bp1 = bp[2 * kq + 1], bg0 = bg[2 * kq], bg1 = bg[2 * kq + 1];
        const float c0 = cc[2 * kq], c1 = cc[2 * kq + 1];
        const float ac = rc[kq], as = rs[kq];
        float* v0 = reinterpret_cast<float*>(&h0);
        float* v1 = reinterpret_cast<float*>(&h1);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float g0 = fmaf(bp0, xpr[c][0], v0[c]), g1 = fmaf(bp1, xpr[c][0], v1[c]);
          const float u0 = bg0 * xr[c][0], u1 = bg1 * xr[c][0];
          const float n0 = fmaf(ac, g0, fmaf(-as, g1, u0));
          const float n1 = fmaf(as, g0, fmaf(ac, g1, u1));
          v0[c] = n0;
          v1[c] = n1;
          yp[c][0] = fmaf(c0, n0, fmaf(c1, n1, yp[c][0]));
        }
        *reinterpret_cast<float4*>(gst + (2 * kq) * P + 4 * q) = h0;
        *reinterpret_cast<float4*>(gst + (2 * kq + 1) * P + 4 * q) = h1;
      }
    } else {
      // h' = alpha Rot h + U (x_prev | x)^T: the 2R-term row sums run on rank
      // pairs as packed two-lane FMAs. X[c][j] = (x_prev | x)[column 4q + c]
      // [ranks 2j, 2j + 1], j < R.
      float2 X[4][R];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int j = 0; j < R / 2; ++j) {
          X[c][j] = make_float2(xpr[c][2 * j], xpr[c][2 * j + 1]);
          X[c][R / 2 + j] = make_float2(xr[c][2 * j], xr[c][2 * j + 1]);
        }
      const float4* U4 = reinterpret_cast<const float4*>(ud);  // R / 2 float4 per row
      const float2* R2 = reinterpret_cast<const float2*>(rd);
      for (int it = tid; ok && it < items; it += kSThreads) {
        const int kq = it / PQ;
        float4 h0 = *reinterpret_cast<const float4*>(sst + (2 * kq) * P + 4 * q);
        float4 h1 = *reinterpret_cast<const float4*>(sst + (2 * kq + 1) * P + 4 * q);
        float2 w0[R], w1[R];
#pragma unroll
        for (int j = 0; j < R / 2; ++j) {
          const float4 t0 = U4[2 * kq * (R / 2) + j], t1 = U4[(2 * kq + 1) * (R / 2) + j];
          w0[2 * j] = make_float2(t0.x, t0.y);
          w0[2 * j + 1] = make_float2(t0.z, t0.w);
          w1[2 * j] = make_float2(t1.x, t1.y);
          w1[2 * j + 1] = make_float2(t1.z, t1.w);
        }
        float c0[R], c1[R];
        ld_row<R>(cd + (2 * kq) * R, c0);
        ld_row<R>(cd + (2 * kq + 1) * R, c1);
        const float2 rot = R2[kq];
        const float ac = rot.x, as = rot.y;
        float* v0 = reinterpret_cast<float*>(&h0);
        float* v1 = reinterpret_cast<float*>(&h1);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float2 s0 = ptx::mul2(w0[0], X[c][0]), s1 = ptx::mul2(w1[0], X[c][0]);
#pragma unroll
          for (int j = 1; j < R; ++j) {
            s0 = ptx::fma2(w0[j], X[c][j], s0);
            s1 = ptx::fma2(w1[j], X[c][j], s1);
          }
          const float n0 = fmaf(ac, v0[c], fmaf(-as, v1[c], s0.x + s0.y));
          const float n1 = fmaf(as, v0[c], fmaf(ac, v1[c], s1.x + s1.y));
          v0[c] = n0;
          v1[c] = n1;
          const float2 n02 = make_float2(n0, n0), n12 = make_float2(n1, n1);
#pragma unroll
          for (int r = 0; r < R; r += 2) {
            const float2 y2 = ptx::fma2(make_float2(c0[r], c0[r + 1]), n02,
                                        ptx::fma2(make_float2(c1[r], c1[r + 1]), n12,
                                                  make_float2(yp[c][r], yp[c][r + 1])));
            yp[c][r] = y2.x;
            yp[c][r + 1] = y2.y;
          }
        }
        *reinterpret_cast<float4*>(gst + (2 * kq) * P + 4 * q) = h0;
        *reinterpret_cast<float4*>(gst + (2 * kq + 1) * P + 4 * q) = h1;
      }
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
        for (int r = 0; r < R; ++r) yred[((warp * 4 + c) * R + r) * (PQ + 1) + q] = yp[c][r];
    }
    __syncthreads();
    if (abort_flag) break;  // uniform: read after the barrier
    // stage s is read: refill it with the unit kStages ahead
    if (tid == 0) {
      const int un = u + kStages * (int)gridDim.x;
      if (un < units) issue(un, s);
    }
    T* out = static_cast<T*>(a.out) + (int64_t)u * P * R;
    for (int i = tid; i < P * R; i += kSThreads) {
      const int pp = i / R, r = i - pp * R;
      const int at = ((pp & 3) * R + r) * (PQ + 1) + (pp >> 2);
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < kSWarps; ++w) acc += yred[w * 4 * R * (PQ + 1) + at];
      st_act(out + i, acc);
    }
  }
  // after an abort, let the copies in flight land before the CTA ends
  if (tid == 0) {
    for (int j = 0; j < kStages; ++j, ++k) {
      const int u = blockIdx.x + k * (int)gridDim.x;
      if (u >= units) break;
      ptx::mbar_wait(&full[k % kStages], (uint32_t)((k / kStages) & 1), kStreamWaitNs);
    }
  }
}

// The streaming kernel's conditions: every per-unit block 16-byte aligned and
// a multiple of 16 bytes, the dt / lambda windows inside their arrays, and
// two CTAs' shared memory on one SM.
bool stream_ok(const DecodeArgs& a, int act, size_t* smem) {
  auto al = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  const int64_t N = a.N, P = a.P, R = a.R;
  if (P % 4 != 0 || 32 % (P / 4) != 0) return false;
  if ((N * P * 4) % 16 || (P * R * act) % 16 || (N * R * act) % 16 || (N / 2 * 4) % 16) return false;
  if ((a.B_bias || a.C_bias) && (N * R * 4) % 16) return false;
  if ((a.batch * a.H) % 4 != 0) return false;
  if (!al(a.state) || !al(a.x) || !al(a.x_prev) || !al(a.B) || !al(a.B_prev) || !al(a.C) ||
      !al(a.theta) || !al(a.B_bias) || !al(a.C_bias) || !al(a.dt) || !al(a.lam))
    return false;
  const StreamLayout L = stream_layout(a, act);
  *smem = stream_smem_bytes(a, L);
  return *smem <= 112 * 1024;
}

int stream_grid(int units) {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      sms = 148;
  }
  const int g = 2 * sms;
  return units < g ? units : g;
}

template <typename T>
cudaError_t launch_stream_t(const DecodeArgs& a, size_t smem, cudaStream_t s) {
  const StreamLayout L = stream_layout(a, (int)sizeof(T));
  const int units = (int)(a.batch * a.H);
  const dim3 grid((unsigned)stream_grid(units));
  cudaError_t e = cudaSuccess;
  switch (a.R) {
    case 1:
      e = cudaFuncSetAttribute(decode_stream_kernel<T, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) decode_stream_kernel<T, 1><<<grid, kSThreads, smem, s>>>(a, L, units);
      break;
    case 2:
      e = cudaFuncSetAttribute(decode_stream_kernel<T, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) decode_stream_kernel<T, 2><<<grid, kSThreads, smem, s>>>(a, L, units);
      break;
    case 4:
      e = cudaFuncSetAttribute(decode_stream_kernel<T, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) decode_stream_kernel<T, 4><<<grid, kSThreads, smem, s>>>(a, L, units);
      break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
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
  size_t smem = 0;
  if (decode_mma_ok(a, bf16)) return launch_decode_mma(a, s);
  if (a.status != nullptr && stream_ok(a, bf16 ? 2 : 4, &smem))
    return bf16 ? launch_stream_t<__nv_bfloat16>(a, smem, s) : launch_stream_t<float>(a, smem, s);
  return bf16 ? launch_t<__nv_bfloat16>(a, s) : launch_t<float>(a, s);
}

}  // namespace m3
