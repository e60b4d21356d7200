// Affine quantisation (load time) and the materialising dequantisation.
//
// Format: MLX affine packed weights -- a uint32 payload of 4- or 8-bit codes,
// low bits first, with one scale and one bias per group of 64 along K
// ("epic: realize low-precision / quantized performance on the OpenXLA (IREE)
// backend", section Context).  Reconstruction is w = q*scale + bias after a
// bit-unpack ("track(upstream-iree): fused dequant->matmul for the packed int8
// bandwidth win", section "What is already in-tree").
//
// Both kernels are HBM-bound elementwise passes; neither is on the per-token
// path.  Rounding is spelled out so the results are bit-identical to a
// correctly rounded host computation:
//   * quantise: f32 subtract and divide with explicit _rn intrinsics (no
//     contraction), rint (ties to even), stored scale/bias rounded with RNE;
//   * dequant: q*scale is exact in every output precision, so a single fused
//     multiply-add in the output precision rounds the exact value once.

#include "device_common.cuh"
#include "qlin_internal.h"

namespace qlin {
namespace {

// One warp per (row, group): a group is 64 consecutive floats, two per lane.
template <int BITS, typename ST>
__global__ void __launch_bounds__(256) quantize_kernel(const float* __restrict__ w,
                                                       int64_t n_groups,
                                                       uint32_t* __restrict__ wq,
                                                       ST* __restrict__ scales,
                                                       ST* __restrict__ biases) {
  constexpr int kPerWord = 32 / BITS;     // codes per word
  constexpr int kLanesPerWord = kPerWord / 2;
  constexpr float kQmax = float((1 << BITS) - 1);
  const int lane = threadIdx.x & 31;
  const int64_t grp = int64_t(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (grp >= n_groups) return;

  const float2 v = reinterpret_cast<const float2*>(w + grp * kGroup)[lane];
  float mn = fminf(v.x, v.y), mx = fmaxf(v.x, v.y);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  const float scale32 = __fdiv_rn(__fsub_rn(mx, mn), kQmax);
  const ST s = Act<ST>::from_f32_rn(scale32);
  const ST b = Act<ST>::from_f32_rn(mn);
  const float sf = Act<ST>::to_f32(s), bf = Act<ST>::to_f32(b);

  uint32_t q0 = 0, q1 = 0;
  if (sf != 0.0f) {
    const float t0 = rintf(__fdiv_rn(__fsub_rn(v.x, bf), sf));
    const float t1 = rintf(__fdiv_rn(__fsub_rn(v.y, bf), sf));
    q0 = static_cast<uint32_t>(fminf(fmaxf(t0, 0.0f), kQmax));
    q1 = static_cast<uint32_t>(fminf(fmaxf(t1, 0.0f), kQmax));
  }
  // element k = 2*lane (+1) sits at position k % kPerWord of word k / kPerWord
  const int pos = (2 * lane) % kPerWord;
  uint32_t part = (q0 << (BITS * pos)) | (q1 << (BITS * (pos + 1)));
#pragma unroll
  for (int o = 1; o < kLanesPerWord; o <<= 1) part |= __shfl_xor_sync(0xffffffffu, part, o);
  if (lane % kLanesPerWord == 0)
    wq[grp * (kGroup / kPerWord) + lane / kLanesPerWord] = part;
  if (lane == 0) {
    scales[grp] = s;
    biases[grp] = b;
  }
}

// Exactly representable code -> storage type.
template <typename T>
__device__ __forceinline__ T code_to(uint32_t q);
template <>
__device__ __forceinline__ __half code_to<__half>(uint32_t q) {
  return __uint2half_rn(q);  // exact for q < 2048
}
template <>
__device__ __forceinline__ __nv_bfloat16 code_to<__nv_bfloat16>(uint32_t q) {
  return __uint2bfloat16_rn(q);  // exact for q < 256
}

// One thread per packed word; writes its kPerWord reconstructed weights.
template <int BITS, typename ST, typename OT>
__global__ void __launch_bounds__(256) dequant_kernel(const uint32_t* __restrict__ wq,
                                                      const ST* __restrict__ scales,
                                                      const ST* __restrict__ biases,
                                                      int64_t n_words, OT* __restrict__ out) {
  constexpr int kPerWord = 32 / BITS;
  constexpr uint32_t kMask = (1u << BITS) - 1u;
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n_words) return;
  const uint32_t word = wq[i];
  const int64_t grp = i / (kGroup / kPerWord);
  const ST s = scales[grp], b = biases[grp];
  OT r[kPerWord];
#pragma unroll
  for (int j = 0; j < kPerWord; ++j) {
    const uint32_t q = (word >> (BITS * j)) & kMask;
    if constexpr (sizeof(OT) == 4) {
      // q*s is exact in f32 (<= 8 + 11 significant bits): one rounding.
      r[j] = __fmaf_rn(float(q), Act<ST>::to_f32(s), Act<ST>::to_f32(b));
    } else {
      r[j] = __hfma(code_to<ST>(q), s, b);  // one rounding in the 16-bit type
    }
  }
  constexpr int kBytes = kPerWord * int(sizeof(OT));
  static_assert(kBytes % 8 == 0, "vector store");
  if constexpr (kBytes >= 16) {
#pragma unroll
    for (int v = 0; v < kBytes / 16; ++v)
      reinterpret_cast<uint4*>(out + i * kPerWord)[v] = reinterpret_cast<const uint4*>(r)[v];
  } else {
    *reinterpret_cast<uint2*>(out + i * kPerWord) = *reinterpret_cast<const uint2*>(r);
  }
}

template <int BITS, typename ST>
qlin_status quantize_t(const float* w, int64_t N, int64_t K, uint32_t* wq, void* scales,
                       void* biases, cudaStream_t st) {
  const int64_t n_groups = N * (K / kGroup);
  const int64_t blocks = (n_groups + 7) / 8;
  quantize_kernel<BITS, ST><<<dim3(unsigned(blocks)), 256, 0, st>>>(
      w, n_groups, wq, static_cast<ST*>(scales), static_cast<ST*>(biases));
  return check_launch("quantize_kernel");
}

template <int BITS, typename ST, typename OT>
qlin_status dequant_t(const uint32_t* wq, const void* scales, const void* biases, int64_t N,
                      int64_t K, void* out, cudaStream_t st) {
  const int64_t n_words = N * K * BITS / 32;
  const int64_t blocks = (n_words + 255) / 256;
  dequant_kernel<BITS, ST, OT><<<dim3(unsigned(blocks)), 256, 0, st>>>(
      wq, static_cast<const ST*>(scales), static_cast<const ST*>(biases), n_words,
      static_cast<OT*>(out));
  return check_launch("dequant_kernel");
}

template <typename ST>
qlin_status dequant_st(const uint32_t* wq, const void* scales, const void* biases, int64_t N,
                       int64_t K, int bits, qlin_dtype out_dtype, void* out, cudaStream_t st) {
  if (out_dtype == QLIN_F32)
    return bits == 4 ? dequant_t<4, ST, float>(wq, scales, biases, N, K, out, st)
                     : dequant_t<8, ST, float>(wq, scales, biases, N, K, out, st);
  return bits == 4 ? dequant_t<4, ST, ST>(wq, scales, biases, N, K, out, st)
                   : dequant_t<8, ST, ST>(wq, scales, biases, N, K, out, st);
}

}  // namespace

qlin_status launch_quantize(const float* w, int64_t N, int64_t K, int bits, qlin_dtype sdtype,
                            uint32_t* wq, void* scales, void* biases, cudaStream_t st) {
  if ((N * (K / kGroup) + 7) / 8 > 0x7fffffff)
    return fail(QLIN_ERR_UNSUPPORTED, "quantize: too many groups");
  if (sdtype == QLIN_F16)
    return bits == 4 ? quantize_t<4, __half>(w, N, K, wq, scales, biases, st)
                     : quantize_t<8, __half>(w, N, K, wq, scales, biases, st);
  return bits == 4 ? quantize_t<4, __nv_bfloat16>(w, N, K, wq, scales, biases, st)
                   : quantize_t<8, __nv_bfloat16>(w, N, K, wq, scales, biases, st);
}

qlin_status launch_dequant(const uint32_t* wq, const void* scales, const void* biases, int64_t N,
                           int64_t K, int bits, qlin_dtype sdtype, qlin_dtype out_dtype,
                           void* w_out, cudaStream_t st) {
  if ((N * K * bits / 32 + 255) / 256 > 0x7fffffff)
    return fail(QLIN_ERR_UNSUPPORTED, "dequant: too many words");
  if (sdtype == QLIN_F16)
    return dequant_st<__half>(wq, scales, biases, N, K, bits, out_dtype, w_out, st);
  return dequant_st<__nv_bfloat16>(wq, scales, biases, N, K, bits, out_dtype, w_out, st);
}

}  // namespace qlin
