// Internal launcher interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace m3 {

struct ScanArgs {
  const void* x;
  const float* dt;
  const float* A;
  const float* lam;
  const void* B;
  const void* C;
  const float* theta;
  const float* B_bias;
  const float* C_bias;
  void* out;
  float* final_state;
  // state entering the first token ([b,H,N,P] fp32, explicit frame, its
  // pending beta term included), or NULL for zero; may alias final_state
  const float* h_init;
  void* workspace;          // device scratch, or NULL (allocated stream-ordered when needed)
  size_t workspace_bytes;
  int64_t batch, L, H, G, P, N;
  int R, Q;
  bool bc_norm;  // B and C arrive un-normalised: BCNorm them in the prologue
  bool f32;      // fp32 activations (the tensor-core fp32 mode), else bf16
};

struct DecodeArgs {
  float* state;
  const void* x;
  const float* dt;
  const float* A;
  const float* lam;
  const void* B_prev;
  const void* x_prev;
  const void* B;
  const void* C;
  const float* theta;
  const float* B_bias;
  const float* C_bias;
  void* out;
  unsigned int* status;  // device word for expired waits (streaming kernel)
  int64_t batch, H, G, P, N;
  int R;
};

// K consecutive decode tokens (x, out [b,K,H,P,R]; dt, lam [b,K,H];
// B, C [b,K,G,N,R]; theta [b,K,G,N/2]; B_prev [b,G,N,R] and x_prev [b,H,P,R]
// of the token before the block, or both NULL).
struct TokensArgs {
  float* state;
  const void* x;
  const float* dt;
  const float* A;
  const float* lam;
  const void* B_prev;
  const void* x_prev;
  const void* B;
  const void* C;
  const float* theta;
  const float* B_bias;
  const float* C_bias;
  void* out;
  unsigned int* status;  // device word for expired waits (tensor-core kernel)
  int64_t batch, K, H, G, P, N;
  int R;
};

// Backward pass of the prefill from a zero state: gradients of
// <y, dy> + <h_final, d_final>. Gradients are fp32; dA, dB, dC, dtheta and the
// bias gradients are accumulated (zeroed by the launcher), the rest written.
struct BwdArgs {
  const void* x;
  const float* dt;
  const float* A;
  const float* lam;
  const void* B;
  const void* C;
  const float* theta;
  const float* B_bias;
  const float* C_bias;
  const void* dy;          // [b,L,H,P,R], act dtype
  const float* d_final;    // [b,H,N,P] or NULL
  float* dx;               // [b,L,H,P,R]
  float* ddt;              // [b,L,H]
  float* dA;               // [H]
  float* dlam;             // [b,L,H]
  float* dB;               // [b,L,G,N,R]
  float* dC;               // [b,L,G,N,R]
  float* dtheta;           // [b,L,G,N/2]
  float* dB_bias;          // [H,N,R] or NULL
  float* dC_bias;          // [H,N,R] or NULL
  int64_t batch, L, H, G, P, N;
  int R;
};

// CUDA-core chunked prefill (any shape whose tiles fit shared memory).
size_t scan_simt_smem_bytes(int64_t N, int64_t P, int R, int Q);
cudaError_t launch_scan_simt(const ScanArgs& a, bool bf16, cudaStream_t s);

// Tensor-core (tcgen05) chunked prefill, bf16 activations.
bool scan_tc_supported(int64_t N, int64_t P, int R, int Q);
// Scratch the tensor-core prefill needs (segmented long sequences), 0 if none.
size_t scan_tc_workspace_bytes(const ScanArgs& a);
cudaError_t launch_scan_tc(const ScanArgs& a, unsigned int* status, cudaStream_t s);

// Prefill continuation: state[b,h] += beta_hat_0 (B_prev + bias) x_prev^T, the
// pending term of the block's first token (beta_hat_0 = (1 - lam_0) dt_0), in
// place, so that the state becomes the explicit-frame entering state.
cudaError_t launch_entry_state(float* state, const void* B_prev, const void* x_prev,
                               const float* dt, const float* lam, const float* B_bias,
                               int64_t batch, int64_t L, int64_t H, int64_t G, int64_t P,
                               int64_t N, int R, bool bf16, cudaStream_t s);

// Decode step.
bool decode_supported(int64_t N, int64_t P, int R);
cudaError_t launch_decode(const DecodeArgs& a, bool bf16, cudaStream_t s);
// bf16, R = 4, P = 64: the rank-R update on the tensor cores (mma.sync).
bool decode_mma_ok(const DecodeArgs& a, bool bf16);
cudaError_t launch_decode_mma(const DecodeArgs& a, cudaStream_t s);

// K decode tokens in one launch, the state held on chip between them.
bool tokens_supported(const TokensArgs& a, int act);
cudaError_t launch_decode_tokens(const TokensArgs& a, bool bf16, cudaStream_t s);
// bf16, R = 4, P = 64: the rank-R updates on the tensor cores (mma.sync).
bool tokens_mma_ok(const TokensArgs& a, bool bf16);
cudaError_t launch_tokens_mma(const TokensArgs& a, cudaStream_t s);

// Fault injection (M3_FAULT=timeout): a kernel whose bounded wait runs out
// after limit_ns, recording the expiry in the status word.
cudaError_t launch_expired_wait(uint64_t limit_ns, cudaStream_t s);

// Backward pass (CUDA cores, state checkpoints in a stream-ordered scratch).
// bf16, P = 64, N in {64, 128}: the chunked backward on the tensor cores
// (mma.sync TF32), with its workspace (bytes) given by the caller.
bool scan_bwd_tc_ok(const BwdArgs& a, bool bf16);
size_t scan_bwd_tc_workspace(const BwdArgs& a);
cudaError_t launch_scan_bwd_tc(const BwdArgs& a, float* ws, cudaStream_t s);
bool scan_bwd_supported(int64_t N, int64_t P, int R);
// ws: device scratch of scan_bwd_workspace_bytes() bytes (16-byte aligned),
// or NULL: allocated and freed on the stream.
size_t scan_bwd_workspace_bytes(const BwdArgs& a, bool bf16);
cudaError_t launch_scan_bwd(const BwdArgs& a, bool bf16, void* ws, cudaStream_t s);

// Device address of this device's status word of expired waits.
cudaError_t status_word(unsigned int** ptr);
cudaError_t read_clear_status(unsigned int* value, cudaStream_t s);

}  // namespace m3
