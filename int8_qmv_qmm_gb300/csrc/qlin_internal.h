// Internal declarations shared by the libqlin translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "qlin.h"

namespace qlin {

// Records a formatted detail message for qlin_last_error() and returns s.
qlin_status fail(qlin_status s, const char* fmt, ...);

// Maps a CUDA runtime error (if any) from the last launch to a status.
qlin_status check_launch(const char* what);

// Number of SMs of the current device (cached per device).
int sm_count();

// Launchers.  Arguments are already validated by the public entry points.
qlin_status launch_quantize(const float* w, int64_t N, int64_t K, int bits, qlin_dtype sdtype,
                            uint32_t* wq, void* scales, void* biases, cudaStream_t st);
qlin_status launch_dequant(const uint32_t* wq, const void* scales, const void* biases, int64_t N,
                           int64_t K, int bits, qlin_dtype sdtype, qlin_dtype out_dtype,
                           void* w_out, cudaStream_t st);
// A linear layer's epilogue: the layer bias (activation dtype [N], or null)
// added before the final rounding, and float32 output instead of the
// activation dtype.
struct Epilogue {
  const void* bias;
  int y_f32;
};

qlin_status launch_qmv(const void* x, const uint32_t* wq, const void* scales, const void* biases,
                       void* y, int64_t M, int64_t N, int64_t K, int bits, qlin_dtype dtype,
                       unsigned flags, const Epilogue& ep, cudaStream_t st);
qlin_status launch_qmm(const void* x, const uint32_t* wq, const void* scales, const void* biases,
                       void* y, int64_t M, int64_t N, int64_t K, int bits, qlin_dtype dtype,
                       unsigned flags, const Epilogue& ep, cudaStream_t st);

// Limits of the chain kernel's waits for an input link.  stalled_link >= 0
// (tests only) makes the readers of that link wait for one row block more
// than it has, so that their wait runs out.
struct ChainWaitOptions {
  unsigned long long dep_wait_ns;
  int stalled_link;
};
constexpr ChainWaitOptions kDefaultChainWaits = {2000000000ull, -1};

qlin_status launch_qmv_chain(const void* x0, const qlin_link* links, int n_links, int bits,
                             qlin_dtype dtype, void* ws, const ChainWaitOptions& wo,
                             cudaStream_t st);
int chain_max_links();

// The number of CTAs qlin_qmv gives each row block (its split of K) for an
// N x K matrix of `bits`-bit codes on a device with `sms` SMs.
int qmv_plan_split(int64_t N, int64_t K, int bits, int sms);

// Read and clear the kernels' device status words (no synchronisation).
cudaError_t qmm_take_device_status(unsigned* flags);
cudaError_t qmv_take_device_status(unsigned* flags);
cudaError_t chain_take_device_status(unsigned* flags);

constexpr int kGroup = 64;

}  // namespace qlin
