// Internal interface between the C-ABI front end (ccv_api.cpp) and the
// kernel launchers (ccv_fwd_*.cu, ccv_update.cu, ccv_bwd_*.cu).  Not
// installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ccv {

// Validated forward-pass arguments.  Pointers address logical element
// [0,...,0]; strides are in elements.
struct FwdArgs {
  const void* x;
  int64_t xs0, xs1, xs2;
  void* out;
  int64_t os0, os1, os2;
  const void* w;
  int64_t ws0, ws1;
  const void* bias;  // may be null
  int64_t bs;
  const int32_t* seq;  // may be null
  int64_t ss0, ss1;
  const void* init;  // may be null
  int64_t is0, is1, is2;
  void* fin;  // may be null
  int64_t fs0, fs1, fs2;
  int64_t B, C, L;
  int silu;  // 0 or 1
  int wdt;   // Dtype of weight and bias (x, out and the states have the kernel's dtype)
};

// Validated decode-step arguments (see ccv_update in ccv.h).
struct UpdArgs {
  const void* x;
  int64_t xs0, xs1, xs2;
  void* out;
  int64_t os0, os1, os2;
  void* state;
  int64_t ss0, ss1, ss2;
  const void* w;
  int64_t ws0, ws1;
  const void* bias;
  int64_t bs;
  int64_t B, C, S;
  int silu;
  int wdt;  // Dtype of weight and bias
};

// Validated backward-pass arguments (see ccv_bwd in ccv.h).  Time is cut
// into n_chunk partitions of `chunk` steps; partition p = b * n_chunk + chunk
// writes its partial parameter-gradient sums to part[(p * (K+1) + k) * C + c]
// (k = K: dbias), or nothing when part is null.
struct BwdArgs {
  const void* x;
  int64_t xs0, xs1, xs2;
  const void* w;
  int64_t ws0, ws1;
  const void* bias;  // may be null
  int64_t bs;
  const int32_t* seq;  // may be null
  int64_t ss0, ss1;
  const void* init;  // may be null
  int64_t is0, is1, is2;
  const void* dout;
  int64_t gs0, gs1, gs2;
  const void* dfin;  // may be null
  int64_t fs0, fs1, fs2;
  void* dx;
  int64_t dxs0, dxs1, dxs2;
  void* dinit;  // may be null
  int64_t dis0, dis1, dis2;
  float* part;  // may be null
  int64_t B, C, L;
  int64_t chunk, n_chunk;
  int silu;  // 0 or 1
  int wdt;   // Dtype of weight and bias
};

// Fixed-order sum of the partials into dweight [C,K] and dbias [C].
struct RedArgs {
  const float* part;
  int64_t P, C;
  void* dw;  // may be null
  int64_t dws0, dws1;
  void* db;  // may be null
  int64_t dbs;
  int wdt;  // Dtype of dweight and dbias
};

// Layout class of (x, dout, dx) and the time partition of the backward pass.
enum BwdClass { kBwdTime = 0, kBwdChan = 1, kBwdOther = 2 };
struct BwdPlan {
  BwdClass cls;
  int64_t chunk, n_chunk;
};

enum Dtype { kF32 = 0, kF16 = 1, kBF16 = 2 };

struct Device {
  int sm_count;
};

// Each launcher enqueues one kernel on `stream` and returns the launch
// status (cudaGetLastError right after the launch).
cudaError_t launch_fwd_time_vec(const FwdArgs& a, int K, Dtype dt, const Device& dev,
                                cudaStream_t stream);
cudaError_t launch_fwd_chlast_vec(const FwdArgs& a, int K, Dtype dt, const Device& dev,
                                  cudaStream_t stream);
cudaError_t launch_fwd_generic(const FwdArgs& a, int K, Dtype dt, const Device& dev,
                               cudaStream_t stream);
// Which any-stride forward kernel launch_fwd_generic picks: lanes along time
// (true: the time stride is the smaller one) or along channels.
bool generic_time_walk(const FwdArgs& a);

// TMA-staged channel-last kernel: needs a 16-byte aligned x with 16-byte
// multiple batch/time strides (and a contiguous, aligned seq_idx row).
bool chlast_tma_eligible(const FwdArgs& a, int dtype_size);
cudaError_t launch_fwd_chlast_tma(const FwdArgs& a, int K, Dtype dt, const Device& dev,
                                  cudaStream_t stream);

cudaError_t launch_update(const UpdArgs& a, int K, Dtype dt, const Device& dev, cudaStream_t stream);

// Backward pass: the plan (a function of the layout class and sizes only),
// the gradient kernels and the partial-sum reduction.
BwdPlan bwd_plan(BwdClass cls, int64_t B, int64_t C, int64_t L);
cudaError_t launch_bwd_generic(const BwdArgs& a, int K, Dtype dt, const Device& dev, cudaStream_t stream);
cudaError_t launch_bwd_time(const BwdArgs& a, int K, Dtype dt, bool strided, const Device& dev,
                            cudaStream_t stream);
cudaError_t launch_bwd_chlast(const BwdArgs& a, int K, Dtype dt, int channel_stride, const Device& dev,
                              cudaStream_t stream);
cudaError_t launch_bwd_reduce(const RedArgs& r, int K, Dtype dt, cudaStream_t stream);

// Fixed scratch of ccv_bwd_noalloc: its size, and its address on the current
// device (cudaGetSymbolAddress; no allocation).
size_t noalloc_scratch_bytes();
cudaError_t noalloc_scratch_address(void** ptr);

// Test of the bounded waits: the next channel-last TMA launch waits at most
// `budget_cycles` per barrier and leaves out the copy of stage `skip_stage`
// of its first warp (one-shot; budget_cycles <= 0 cancels).
void set_chlast_wait_test(long long budget_cycles, long long skip_stage);

// Fault words of the kernels with bounded barrier waits (read and cleared;
// synchronous).  Non-zero means a wait ran out of budget.
unsigned read_and_clear_fault_chlast_tma();

}  // namespace ccv
