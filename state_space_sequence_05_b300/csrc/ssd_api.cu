// ssd_api.cu -- the extern "C" boundary of libssd_b300.so: argument checks,
// workspace sizing and dispatch to the kernels.  See include/ssd.h for the
// contract of each entry point.
#include <cuda_runtime.h>
#include <string.h>
#include <stdint.h>

#include <atomic>
#include <cstdlib>

#include "ssd.h"
#include "ssd_internal.h"

namespace {

std::atomic<uint64_t> g_launches{0};
// Test hook (ssd_test_set_forward_wait): bound on every device wait of the
// pipelined tensor-core forward and a unit that never publishes its state.
std::atomic<unsigned long long> g_wait_ns{0};
std::atomic<int> g_hold_unit{-1};

}  // namespace

void ssd::count_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

namespace {

using ssd::FwdArgs;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool dstate_ok(int n) { return n == 16 || n == 32 || n == 64 || n == 128 || n == 256; }

// Shape/pointer checks shared by the forward entry point and its workspace
// query.  Pointers are checked only when `check_ptrs`.
ssd_status_t check_fwd(const FwdArgs& a, bool check_ptrs) {
  if (a.dtype != SSD_DT_F32 && a.dtype != SSD_DT_BF16) return SSD_ERR_INVALID;
  if (a.batch < 0 || a.seqlen < 0 || a.H <= 0 || a.P <= 0 || a.N <= 0 || a.G <= 0)
    return SSD_ERR_INVALID;
  if (a.H % a.G != 0) return SSD_ERR_INVALID;
  if ((long long)a.batch * a.seqlen >= (1LL << 31)) return SSD_ERR_UNSUPPORTED;
  if (a.Q != 64 && a.Q != 128 && a.Q != 256) return SSD_ERR_UNSUPPORTED;
  if (a.P > 128 || !dstate_ok(a.N)) return SSD_ERR_UNSUPPORTED;
  if (a.cu) {
    if (a.batch != 1 || a.nseq < 0) return SSD_ERR_INVALID;
    if (a.nseq == 0 && a.seqlen != 0) return SSD_ERR_INVALID;
  }
  if (!check_ptrs) return SSD_OK;
  const long long ntok = (long long)a.batch * a.seqlen;
  if (ntok > 0 && (!a.x || !a.dt || !a.B || !a.C || !a.y)) return SSD_ERR_INVALID;
  if (!a.A) return SSD_ERR_INVALID;
  if (!aligned16(a.x) || !aligned16(a.B) || !aligned16(a.C) || !aligned16(a.y))
    return SSD_ERR_INVALID;
  if (!aligned16(a.init) || !aligned16(a.final_states)) return SSD_ERR_INVALID;
  return SSD_OK;
}

// Which tensor-core forward runs the plain (no fused-epilogue) calls:
// SSD_TC_KERNEL=fused (the default: one kernel with the segment hand-off
// inside), =split (decay tables, segment states, state passing and outputs
// as separate kernels) or =pipelined (the fused design with a deeper
// operand pipeline).
enum class TcKernel { kFused, kSplit, kPipelined };
TcKernel tc_kernel() {
  const char* e = getenv("SSD_TC_KERNEL");
  if (e && strcmp(e, "split") == 0) return TcKernel::kSplit;
  if (e && strcmp(e, "pipelined") == 0) return TcKernel::kPipelined;
  return TcKernel::kFused;
}

size_t fwd_workspace(const FwdArgs& a) {
  if (a.nseq == 0) return 0;
  // any of the tensor-core kernels may run a tensor-core shape (the fused-
  // epilogue options always take the fused kernel): enough for each
  if (ssd::tc_supported(a)) {
    size_t w = ssd::tc_workspace_bytes(a);
    const size_t t2 = ssd::tc2_workspace_bytes(a), t3 = ssd::tc3_workspace_bytes(a);
    if (t2 > w) w = t2;
    if (t3 > w) w = t3;
    return w;
  }
  return ssd::simt_workspace_bytes(a);
}

}  // namespace

ssd_status_t ssd::check_fwd_args(const FwdArgs& a, bool check_ptrs) {
  return check_fwd(a, check_ptrs);
}

extern "C" {

const char* ssd_status_string(ssd_status_t s) {
  switch (s) {
    case SSD_OK: return "ok";
    case SSD_ERR_INVALID: return "invalid argument";
    case SSD_ERR_UNSUPPORTED: return "unsupported shape or option";
    case SSD_ERR_CUDA: return "CUDA runtime error";
    case SSD_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

int ssd_version(void) { return 100; }

uint64_t ssd_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

size_t ssd_chunk_scan_fwd_workspace_size(int batch, int seqlen, int nheads, int headdim,
                                         int dstate, int ngroups, int chunk_size,
                                         ssd_dtype_t in_dtype, int varlen, int nseq) {
  static const int32_t kDummy = 0;
  FwdArgs a{};
  a.batch = batch;
  a.seqlen = seqlen;
  a.H = nheads;
  a.P = headdim;
  a.N = dstate;
  a.G = ngroups;
  a.Q = chunk_size;
  a.dtype = in_dtype;
  a.cu = varlen ? &kDummy : nullptr;  // only its presence matters here
  a.nseq = varlen ? nseq : batch;
  if (check_fwd(a, false) != SSD_OK) return (size_t)-1;
  return fwd_workspace(a);
}

ssd_status_t ssd_chunk_scan_fwd(const void* x, const void* dt, const float* A, const void* B,
                                const void* C, const float* D, int batch, int seqlen,
                                int nheads, int headdim, int dstate, int ngroups, int chunk_size,
                                ssd_dtype_t in_dtype, const float* init_states,
                                const int32_t* cu_seqlens, int nseq, float* y,
                                float* final_states, void* workspace, size_t workspace_bytes,
                                int32_t* dev_status, void* stream) {
  return ssd_chunk_scan_fwd_ex(x, dt, A, B, C, D, batch, seqlen, nheads, headdim, dstate, ngroups,
                               chunk_size, in_dtype, init_states, cu_seqlens, nseq, y,
                               final_states, workspace, workspace_bytes, dev_status, stream,
                               nullptr);
}

ssd_status_t ssd_chunk_scan_fwd_ex(const void* x, const void* dt, const float* A, const void* B,
                                   const void* C, const float* D, int batch, int seqlen,
                                   int nheads, int headdim, int dstate, int ngroups,
                                   int chunk_size, ssd_dtype_t in_dtype, const float* init_states,
                                   const int32_t* cu_seqlens, int nseq, void* y,
                                   float* final_states, void* workspace, size_t workspace_bytes,
                                   int32_t* dev_status, void* stream,
                                   const ssd_fwd_epilogue_t* epilogue) {
  FwdArgs a{};
  a.x = x;
  a.dt = dt;
  a.A = A;
  a.B = B;
  a.C = C;
  a.D = D;
  a.batch = batch;
  a.seqlen = seqlen;
  a.H = nheads;
  a.P = headdim;
  a.N = dstate;
  a.G = ngroups;
  a.Q = chunk_size;
  a.dtype = in_dtype;
  a.init = init_states;
  a.cu = cu_seqlens;
  a.nseq = cu_seqlens ? nseq : batch;
  a.y = static_cast<float*>(y);
  a.final_states = final_states;
  if (epilogue) {
    a.dt_bias = epilogue->dt_bias;
    a.dt_softplus = epilogue->dt_softplus != 0;
    a.z = epilogue->z;
    a.y_bf16 = epilogue->y_bf16 != 0;
  }
  a.ws = workspace;
  a.ws_bytes = workspace_bytes;
  a.dev_status = dev_status;
  a.stream = static_cast<cudaStream_t>(stream);
  ssd_status_t st = check_fwd(a, true);
  if (st != SSD_OK) return st;
  const bool fused = a.dt_softplus || a.z || a.y_bf16;
  if (fused) {
    // the fused epilogue exists on the tensor-core kernel only
    if (!ssd::tc_supported(a)) return SSD_ERR_UNSUPPORTED;
    if (!aligned16(a.z)) return SSD_ERR_INVALID;
  }
  const size_t need = fwd_workspace(a);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need ||
                   (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
    return SSD_ERR_INVALID;
  if (dev_status && cudaMemsetAsync(dev_status, 0, sizeof(int32_t), a.stream) != cudaSuccess)
    return SSD_ERR_CUDA;
  if (a.nseq == 0) return SSD_OK;
  const unsigned long long w = g_wait_ns.load(std::memory_order_relaxed);
  const unsigned long long wait_ns = w ? w : 2000000000ull;
  const int hold = g_hold_unit.load(std::memory_order_relaxed);
  const TcKernel k = tc_kernel();
  if (k == TcKernel::kSplit && ssd::tc3_supported(a)) return ssd::tc3_forward(a, wait_ns, hold);
  if (k == TcKernel::kPipelined && ssd::tc2_supported(a)) return ssd::tc2_forward(a, wait_ns, hold);
  return ssd::tc_supported(a) ? ssd::tc_forward(a, wait_ns, hold) : ssd::simt_forward(a);
}

void ssd_test_set_forward_wait(unsigned long long wait_ns, int hold_unit) {
  g_wait_ns.store(wait_ns, std::memory_order_relaxed);
  g_hold_unit.store(hold_unit, std::memory_order_relaxed);
}

ssd_status_t ssd_state_update(float* state, const void* x, const void* dt, const float* A,
                              const void* B, const void* C, const float* D, int batch,
                              int nheads, int headdim, int dstate, int ngroups,
                              ssd_dtype_t in_dtype, float* y, void* stream) {
  if (in_dtype != SSD_DT_F32 && in_dtype != SSD_DT_BF16) return SSD_ERR_INVALID;
  if (batch < 0 || nheads <= 0 || headdim <= 0 || dstate <= 0 || ngroups <= 0)
    return SSD_ERR_INVALID;
  if (nheads % ngroups != 0) return SSD_ERR_INVALID;
  if (!dstate_ok(dstate)) return SSD_ERR_UNSUPPORTED;
  if ((long long)batch * nheads >= (1LL << 31)) return SSD_ERR_UNSUPPORTED;
  if (batch == 0) return SSD_OK;
  if (!state || !x || !dt || !A || !B || !C || !y) return SSD_ERR_INVALID;
  if (!aligned16(state) || !aligned16(B) || !aligned16(C)) return SSD_ERR_INVALID;
  return ssd::decode_step(state, x, dt, A, B, C, D, batch, nheads, headdim, dstate, ngroups,
                          in_dtype, y, static_cast<cudaStream_t>(stream));
}

namespace {

// shapes of the backward: batch mode, P * N up to 16384 (the state and its
// adjoint live in shared memory)
ssd_status_t check_bwd(ssd_dtype_t dtype, int batch, int seqlen, int H, int P, int N, int G) {
  if (dtype != SSD_DT_F32 && dtype != SSD_DT_BF16) return SSD_ERR_INVALID;
  if (batch < 0 || seqlen < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G) return SSD_ERR_INVALID;
  if ((long long)P * N > 16384 || (long long)batch * H >= (1LL << 31) ||
      (long long)batch * seqlen >= (1LL << 31))
    return SSD_ERR_UNSUPPORTED;
  return SSD_OK;
}

}  // namespace

size_t ssd_chunk_scan_bwd_workspace_size(int batch, int seqlen, int nheads, int headdim,
                                         int dstate, int ngroups, ssd_dtype_t in_dtype) {
  if (check_bwd(in_dtype, batch, seqlen, nheads, headdim, dstate, ngroups) != SSD_OK)
    return (size_t)-1;
  return ssd::bwd_workspace_bytes(batch, seqlen, nheads, headdim, dstate);
}

ssd_status_t ssd_chunk_scan_bwd(const void* x, const void* dt, const float* A, const void* B,
                                const void* C, const float* D, int batch, int seqlen, int nheads,
                                int headdim, int dstate, int ngroups, ssd_dtype_t in_dtype,
                                const float* init_states, const float* dy, const float* dfinal,
                                float* dx, float* ddt, float* dA, float* dB, float* dC, float* dD,
                                float* dinit, void* workspace, size_t workspace_bytes,
                                int32_t* dev_status, void* stream) {
  ssd_status_t st = check_bwd(in_dtype, batch, seqlen, nheads, headdim, dstate, ngroups);
  if (st != SSD_OK) return st;
  if (batch == 0) return SSD_OK;
  if (!A || !dA) return SSD_ERR_INVALID;
  if (seqlen > 0 && (!x || !dt || !B || !C || !dy || !dx || !ddt || !dB || !dC))
    return SSD_ERR_INVALID;
  const size_t need = ssd::bwd_workspace_bytes(batch, seqlen, nheads, headdim, dstate);
  if (seqlen > 0 && (workspace == nullptr || workspace_bytes < need ||
                     (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
    return SSD_ERR_INVALID;
  ssd::BwdArgs a{};
  a.x = x;
  a.dt = dt;
  a.B = B;
  a.C = C;
  a.A = A;
  a.D = D;
  a.init = init_states;
  a.dy = dy;
  a.dfinal = dfinal;
  a.dx = dx;
  a.ddt = ddt;
  a.dA = dA;
  a.dB = dB;
  a.dC = dC;
  a.dD = dD;
  a.dinit = dinit;
  a.batch = batch;
  a.seqlen = seqlen;
  a.H = nheads;
  a.P = headdim;
  a.N = dstate;
  a.G = ngroups;
  a.dtype = in_dtype;
  a.ws = workspace;
  a.dev_status = dev_status;
  a.stream = static_cast<cudaStream_t>(stream);
  if (dev_status && cudaMemsetAsync(dev_status, 0, sizeof(int32_t), a.stream) != cudaSuccess)
    return SSD_ERR_CUDA;
  return ssd::bwd(a);
}

namespace {

// The forward's arguments for a states-only call: C and y are not read by
// the segment-state kernels; the CUDA-core path computes y into scratch
// (with B standing in for C, whose values then do not matter).
FwdArgs states_args(const void* x, const void* dt, const float* A, const void* B, int batch,
                    int seqlen, int nheads, int headdim, int dstate, int ngroups, int chunk_size,
                    ssd_dtype_t in_dtype, const float* init_states, const int32_t* cu_seqlens,
                    int nseq, float* final_states) {
  FwdArgs a{};
  a.x = x;
  a.dt = dt;
  a.A = A;
  a.B = B;
  a.C = B;
  a.batch = batch;
  a.seqlen = seqlen;
  a.H = nheads;
  a.P = headdim;
  a.N = dstate;
  a.G = ngroups;
  a.Q = chunk_size;
  a.dtype = in_dtype;
  a.init = init_states;
  a.cu = cu_seqlens;
  a.nseq = cu_seqlens ? nseq : batch;
  a.final_states = final_states;
  return a;
}

// Scratch of a states-only call: the split tensor-core kernels' workspace,
// or the CUDA-core forward's plus room for the dropped y.
size_t states_workspace(const FwdArgs& a, size_t* y_offset) {
  if (a.nseq == 0) return 0;
  if (ssd::tc3_supported(a)) return ssd::tc3_workspace_bytes(a);
  const size_t w = ssd::align256(ssd::simt_workspace_bytes(a));
  *y_offset = w;
  return w + ssd::align256(sizeof(float) * (size_t)a.batch * a.seqlen * a.H * a.P);
}

}  // namespace

size_t ssd_chunk_scan_states_workspace_size(int batch, int seqlen, int nheads, int headdim,
                                            int dstate, int ngroups, int chunk_size,
                                            ssd_dtype_t in_dtype, int varlen, int nseq) {
  static const int32_t kDummy = 0;
  FwdArgs a = states_args(nullptr, nullptr, nullptr, nullptr, batch, seqlen, nheads, headdim,
                          dstate, ngroups, chunk_size, in_dtype, nullptr,
                          varlen ? &kDummy : nullptr, nseq, nullptr);
  if (check_fwd(a, false) != SSD_OK) return (size_t)-1;
  size_t yoff = 0;
  return states_workspace(a, &yoff);
}

ssd_status_t ssd_chunk_scan_states(const void* x, const void* dt, const float* A, const void* B,
                                   int batch, int seqlen, int nheads, int headdim, int dstate,
                                   int ngroups, int chunk_size, ssd_dtype_t in_dtype,
                                   const float* init_states, const int32_t* cu_seqlens, int nseq,
                                   float* final_states, void* workspace, size_t workspace_bytes,
                                   int32_t* dev_status, void* stream) {
  FwdArgs a = states_args(x, dt, A, B, batch, seqlen, nheads, headdim, dstate, ngroups,
                          chunk_size, in_dtype, init_states, cu_seqlens, nseq, final_states);
  a.dev_status = dev_status;
  a.stream = static_cast<cudaStream_t>(stream);
  ssd_status_t st = check_fwd(a, false);
  if (st != SSD_OK) return st;
  const long long ntok = (long long)a.batch * a.seqlen;
  if (!final_states || !A) return SSD_ERR_INVALID;
  if (ntok > 0 && (!x || !dt || !B)) return SSD_ERR_INVALID;
  if (!aligned16(x) || !aligned16(B) || !aligned16(init_states) || !aligned16(final_states))
    return SSD_ERR_INVALID;
  size_t yoff = 0;
  const size_t need = states_workspace(a, &yoff);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need ||
                   (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
    return SSD_ERR_INVALID;
  a.ws = workspace;
  a.ws_bytes = workspace_bytes;
  if (dev_status && cudaMemsetAsync(dev_status, 0, sizeof(int32_t), a.stream) != cudaSuccess)
    return SSD_ERR_CUDA;
  if (a.nseq == 0) return SSD_OK;
  const unsigned long long w = g_wait_ns.load(std::memory_order_relaxed);
  const unsigned long long wait_ns = w ? w : 2000000000ull;
  if (ssd::tc3_supported(a)) return ssd::tc3_states(a, wait_ns);
  a.y = reinterpret_cast<float*>(static_cast<char*>(workspace) + yoff);
  a.ws_bytes = yoff;
  return ssd::simt_forward(a);
}

ssd_status_t ssd_segment_decay(const void* dt, const float* A, int batch, int seqlen, int nheads,
                               ssd_dtype_t in_dtype, float* decay, void* stream) {
  if (in_dtype != SSD_DT_F32 && in_dtype != SSD_DT_BF16) return SSD_ERR_INVALID;
  if (batch < 0 || seqlen < 0 || nheads <= 0) return SSD_ERR_INVALID;
  if ((long long)batch * nheads >= (1LL << 31) || (long long)batch * seqlen >= (1LL << 31))
    return SSD_ERR_UNSUPPORTED;
  if (batch == 0) return SSD_OK;
  if (!A || !decay || (seqlen > 0 && !dt)) return SSD_ERR_INVALID;
  return ssd::segment_decay(dt, A, batch, seqlen, nheads, in_dtype, decay,
                            static_cast<cudaStream_t>(stream));
}

ssd_status_t ssd_segment_combine(const float* decay, const float* states,
                                 const float* init_states, int nsegments, int batch, int nheads,
                                 int headdim, int dstate, float* states_in, void* stream) {
  if (nsegments < 0 || batch < 0 || nheads <= 0 || headdim <= 0 || dstate <= 0)
    return SSD_ERR_INVALID;
  if ((long long)batch * nheads >= (1LL << 31)) return SSD_ERR_UNSUPPORTED;
  if (batch == 0) return SSD_OK;
  if (!states_in || (nsegments > 0 && (!decay || !states))) return SSD_ERR_INVALID;
  return ssd::segment_combine(decay, states, init_states, nsegments, batch, nheads, headdim,
                              dstate, states_in, static_cast<cudaStream_t>(stream));
}

ssd_status_t ssd_selective_scan_fwd(const void* x, const void* dt, const float* A, const void* B,
                                    const void* C, const float* D, const float* init_states,
                                    int batch, int seqlen, int dmodel, int dstate,
                                    ssd_dtype_t in_dtype, float* y, float* final_states,
                                    void* stream) {
  if (in_dtype != SSD_DT_F32 && in_dtype != SSD_DT_BF16) return SSD_ERR_INVALID;
  if (batch < 0 || seqlen < 0 || dmodel <= 0 || dstate <= 0) return SSD_ERR_INVALID;
  if (!dstate_ok(dstate) || batch > 65535) return SSD_ERR_UNSUPPORTED;
  if ((long long)batch * seqlen * dmodel >= (1LL << 40)) return SSD_ERR_UNSUPPORTED;
  if (batch == 0) return SSD_OK;
  if (!A) return SSD_ERR_INVALID;
  if (seqlen > 0 && (!x || !dt || !B || !C || !y)) return SSD_ERR_INVALID;
  if (!aligned16(B) || !aligned16(C)) return SSD_ERR_INVALID;
  return ssd::s6_forward(x, dt, A, B, C, D, init_states, batch, seqlen, dmodel, dstate,
                         in_dtype, y, final_states, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
