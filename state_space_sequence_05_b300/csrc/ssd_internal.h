// ssd_internal.h -- declarations shared between the library's translation
// units (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ssd.h"

namespace ssd {

struct FwdArgs {
  const void* x;
  const void* dt;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  int batch, seqlen, H, P, N, G, Q;
  ssd_dtype_t dtype;
  const float* init;
  const int32_t* cu;
  int nseq;  // sequences: cu ? nseq : batch
  float* y;  // bfloat16 storage when y_bf16
  float* final_states;
  // fused epilogue options (ssd_fwd_epilogue_t); zero = none
  const float* dt_bias;
  int dt_softplus;
  const void* z;
  int y_bf16;
  void* ws;
  size_t ws_bytes;
  int32_t* dev_status;
  cudaStream_t stream;
};

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Launch accounting behind ssd_kernel_launches(): every launch site calls
// this once per kernel it launches.
void count_launches(unsigned n);

// Upper bound on the number of `q`-token chunks over all sequences.
inline long long max_chunks(int batch, int seqlen, int q, bool varlen, int nseq) {
  long long per = (seqlen + q - 1) / q;
  return varlen ? per + nseq : (long long)batch * per;
}

// Sequence plan: offs[0..nseq] chunk offsets plus one status word.
inline size_t plan_bytes(int nseq) { return align256(sizeof(int32_t) * (size_t(nseq) + 2)); }

// Launch the plan kernel: chunk offsets of `q`-token chunks per sequence
// into `offs`, with cu_seqlens validation.  When given, `*ticket` is zeroed
// and final_states[s] = init[s] (or 0) for sequences without tokens.
cudaError_t launch_plan(const int32_t* cu, int seqlen_rows, int seqlen_total, int nseq, int q,
                        int32_t* offs, int32_t* dev_status, cudaStream_t stream,
                        int* ticket = nullptr, const float* init = nullptr,
                        float* final_states = nullptr, int H = 0, int PN = 0);

// Host-side argument checks of ssd_chunk_scan_fwd (pointers only when
// `check_ptrs`), shared with the allocation-free entry point.
ssd_status_t check_fwd_args(const FwdArgs& a, bool check_ptrs);

// CUDA-core (SIMT) chunked forward: any supported shape, fp32 or bf16 in.
size_t simt_workspace_bytes(const FwdArgs& a);
ssd_status_t simt_forward(const FwdArgs& a);

// tcgen05 tensor-core forward: bf16 in, headdim 64, dstate 128, with the
// fused-epilogue options.  Every device wait is bounded by `wait_ns`;
// `hold_unit` >= 0 names a work unit that never publishes its segment end
// state (a test hook: its successor's wait runs out and the call reports
// SSD_ERR_TIMEOUT).
bool tc_supported(const FwdArgs& a);
size_t tc_workspace_bytes(const FwdArgs& a);
ssd_status_t tc_forward(const FwdArgs& a, unsigned long long wait_ns, int hold_unit);

// Pipelined tcgen05 forward (the same shapes, no fused-epilogue options).
// Every device wait is bounded by `wait_ns`; `hold_unit` >= 0 names a work
// unit that never publishes its segment end state (a test hook: its
// successor's wait runs out and the call reports SSD_ERR_TIMEOUT).
bool tc2_supported(const FwdArgs& a);
size_t tc2_workspace_bytes(const FwdArgs& a);
ssd_status_t tc2_forward(const FwdArgs& a, unsigned long long wait_ns, int hold_unit);

// Three-kernel tcgen05 forward (segment states, state passing, outputs; the
// same shapes, no fused-epilogue options).  Every device wait is bounded by
// `wait_ns`; `hold_unit` >= 0 names a work unit whose first decay mask is
// never published (a test hook: the MMA issuer's wait runs out and the call
// reports SSD_ERR_TIMEOUT).
bool tc3_supported(const FwdArgs& a);
size_t tc3_workspace_bytes(const FwdArgs& a);
ssd_status_t tc3_forward(const FwdArgs& a, unsigned long long wait_ns, int hold_unit);
// The segment-state and state-passing kernels alone: final_states (and the
// segments' entering states in the workspace) without y.  Same workspace
// as tc3_forward; a.C, a.D and a.y are not used.
ssd_status_t tc3_states(const FwdArgs& a, unsigned long long wait_ns);

// Mamba-1 selective scan (a decay per channel and state), one launch.
ssd_status_t s6_forward(const void* x, const void* dt, const float* A, const void* B,
                        const void* C, const float* D, const float* init, int batch, int L,
                        int Dm, int N, ssd_dtype_t dtype, float* y, float* final_states,
                        cudaStream_t stream);

// Backward of the forward (batch mode).
struct BwdArgs {
  const void *x, *dt, *B, *C;
  const float *A, *D, *init, *dy, *dfinal;
  float *dx, *ddt, *dA, *dB, *dC, *dD, *dinit;
  int batch, seqlen, H, P, N, G;
  ssd_dtype_t dtype;
  void* ws;
  int32_t* dev_status;  // may be null
  cudaStream_t stream;
};
size_t bwd_workspace_bytes(int batch, int T, int H, int P, int N);
ssd_status_t bwd(const BwdArgs& a);
// The chunked backward (headdim <= 64, dstate <= 128); `bwd` takes it for
// those shapes after zeroing the summed gradients, and the step-by-step
// backward otherwise.
bool bwd_chunked_supported(int P, int N);
size_t bwd_chunked_workspace_bytes(int batch, int T, int H, int P, int N);
ssd_status_t bwd_chunked(const BwdArgs& a);
// dA, ddt, dD, dB and dC zeroed on the call's stream (the gradients that
// the backward kernels accumulate).
cudaError_t bwd_zero_grads(const BwdArgs& a);

// Context parallelism: per-slice log-decay sums and the composition of the
// slices' affine state maps.
ssd_status_t segment_decay(const void* dt, const float* A, int batch, int T, int H,
                           ssd_dtype_t dtype, float* a, cudaStream_t stream);
ssd_status_t segment_combine(const float* a, const float* S, const float* init, int R, int batch,
                             int H, int P, int N, float* h_in, cudaStream_t stream);

// Decode step.
ssd_status_t decode_step(float* state, const void* x, const void* dt, const float* A,
                         const void* B, const void* C, const float* D, int batch, int H, int P,
                         int N, int G, ssd_dtype_t dtype, float* y, cudaStream_t stream);

}  // namespace ssd
